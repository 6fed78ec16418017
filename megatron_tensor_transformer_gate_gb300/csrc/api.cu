// api.cu — the C ABI of include/tp.h: argument validation, workspace carving
// and the launch sequence of each block.  Every compute call only enqueues
// kernels on the caller's stream; nothing here allocates memory.
#include <algorithm>
#include <atomic>
#include <cfenv>
#include <cmath>
#include <cstring>
#include <mutex>

#include "../../include/tp.h"
#include "attention.h"
#include "common.cuh"
#include "elementwise.h"
#include "gemm.h"
#include "profile.h"

#include <vector>

namespace tp {

// Device status word (see common.cuh); kernels receive its address.
__device__ unsigned g_status[4];

namespace {

std::atomic<uint64_t> g_launches{0};
constexpr int kMaxDevices = 64;
int g_sms[kMaxDevices];
unsigned* g_status_ptr[kMaxDevices];
std::mutex g_dev_mu;

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return -1;
  return dev;
}

}  // namespace

void count_launch(int n) { g_launches.fetch_add((uint64_t)n); }

int device_sm_count() {
  const int dev = current_device();
  if (dev < 0) return 1;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (g_sms[dev] == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) !=
            cudaSuccess ||
        v <= 0)
      v = 1;
    g_sms[dev] = v;
  }
  return g_sms[dev];
}

unsigned* device_status_ptr() {
  const int dev = current_device();
  if (dev < 0) return nullptr;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  if (g_status_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<unsigned*>(p);
  }
  return g_status_ptr[dev];
}

// ---------------------------------------------------------------- profiler --
namespace {
struct ProfRec {
  int family;
  double flops, bytes;
};
struct Profiler {
  std::mutex mu;
  bool enabled = false;
  int max = 0, used = 0;
  std::vector<cudaEvent_t> ev;  // 2 per slot: start, end
  std::vector<ProfRec> rec;
};
Profiler g_prof;
}  // namespace

ProfScope::ProfScope(void* s, int family, double flops, double bytes)
    : slot(-1), stream(s) {
  std::lock_guard<std::mutex> lk(g_prof.mu);
  if (!g_prof.enabled || g_prof.used >= g_prof.max) return;
  slot = g_prof.used++;
  g_prof.rec[slot] = ProfRec{family, flops, bytes};
  cudaEventRecord(g_prof.ev[2 * slot], static_cast<cudaStream_t>(s));
}

ProfScope::~ProfScope() {
  if (slot >= 0)
    cudaEventRecord(g_prof.ev[2 * slot + 1], static_cast<cudaStream_t>(stream));
}

}  // namespace tp

using namespace tp;

namespace {

// Sequential carving of a caller buffer into 256-byte aligned regions; with a
// null base it only measures.
struct Carver {
  char* base;
  size_t off = 0;
  explicit Carver(void* b) : base(static_cast<char*>(b)) {}
  void* take(size_t bytes) {
    const size_t o = (off + 255) & ~size_t(255);
    off = o + bytes;
    return base ? base + o : nullptr;
  }
};

bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}
bool opt_aligned(const void* p) { return p == nullptr || aligned16(p); }

size_t elem_size(int32_t dtype) { return dtype == TP_F32 ? 4 : 2; }

std::atomic<int> g_last_cuda_error{0};

tp_status cuda_status(int err) {
  if (err == 0) return TP_OK;
  g_last_cuda_error.store(err);
  return TP_ERR_CUDA;
}

DropoutSpec make_dropout(float p, uint64_t seed) {
  DropoutSpec d;
  if (p > 0.0f) {
    d.enabled = 1;
    // thr = round(p·2^24), ties to even (the current rounding mode)
    d.thr = (uint32_t)std::nearbyint((double)p * 16777216.0);
    d.scale = 1.0f / (1.0f - p);
    d.seed = seed;
  }
  return d;
}

int run_gemm(const GemmProblem& g, tp_stream s) {
  if (g.dtype == TP_BF16 || g.dtype == TP_FP8)
    return launch_gemm_tc(g, s, device_status_ptr());
  return launch_gemm_simt(g, s);
}

// The dtype tensors are stored in: FP8 mode keeps bf16 storage.
int32_t storage(int32_t dtype) { return dtype == TP_FP8 ? TP_BF16 : dtype; }

template <typename F>
tp_status guarded(F&& f) {
  try {
    return f();
  } catch (...) {
    return TP_ERR_CUDA;
  }
}

// ------------------------------------------------------------------- MLP --
tp_status check_mlp(const tp_mlp_desc* d) {
  if (d == nullptr) return TP_ERR_NULL;
  if (d->dtype != TP_F32 && d->dtype != TP_BF16 && d->dtype != TP_FP8)
    return TP_ERR_DTYPE;
  if (d->act != TP_GELU && d->act != TP_SWIGLU) return TP_ERR_DTYPE;
  if (d->mode != TP_REDUCE_FUSED && d->mode != TP_REDUCE_MATERIALISED &&
      d->mode != TP_REDUCE_OVERLAP && d->mode != TP_REDUCE_SP)
    return TP_ERR_DTYPE;
  if (d->T < 1 || d->h < 8 || d->h_ffn < 8 || d->n < 1) return TP_ERR_SHAPE;
  if (d->T > (1 << 30) || d->h > (1 << 20) || d->h_ffn > (1 << 24))
    return TP_ERR_SHAPE;
  if (d->h % 8 || d->h_ffn % d->n || (d->h_ffn / d->n) % 8) return TP_ERR_SHAPE;
  if (d->dtype == TP_FP8 && (d->h % 16 || (d->h_ffn / d->n) % 16))
    return TP_ERR_SHAPE;   // E4M3 rows: multiples of 16 bytes
  if (!(d->dropout_p >= 0.0f && d->dropout_p < 1.0f)) return TP_ERR_ARG;
  return TP_OK;
}

struct MlpFwdLayout {
  void *h_or_g = nullptr, *u = nullptr, *a = nullptr, *partials = nullptr;
  // FP8 mode: E4M3 copies, scales (X, W1, A, W2) and amax scratch words
  void *xq = nullptr, *w1q = nullptr, *aq = nullptr, *w2q = nullptr;
  float* scales = nullptr;
  unsigned* amax = nullptr;
  size_t bytes = 0;
};

MlpFwdLayout mlp_fwd_layout(const tp_mlp_desc* d, void* ws) {
  MlpFwdLayout L;
  Carver c(ws);
  const size_t es = elem_size(d->dtype);
  const size_t tf = (size_t)d->T * (size_t)d->h_ffn * es;
  L.h_or_g = c.take(tf);
  if (d->act == TP_SWIGLU) L.u = c.take(tf);
  L.a = c.take(tf);
  if (d->mode != TP_REDUCE_FUSED)
    L.partials = c.take((size_t)d->n * (size_t)d->T * (size_t)d->h * es);
  if (d->dtype == TP_FP8) {
    const size_t w1rows = d->act == TP_SWIGLU ? 2 * d->h_ffn : d->h_ffn;
    L.xq = c.take((size_t)d->T * (size_t)d->h);
    L.w1q = c.take(w1rows * (size_t)d->h);
    L.aq = c.take((size_t)d->T * (size_t)d->h_ffn);
    L.w2q = c.take((size_t)d->h * (size_t)d->h_ffn);
    L.scales = static_cast<float*>(c.take(4 * sizeof(float)));
    L.amax = static_cast<unsigned*>(c.take(4 * sizeof(unsigned)));
  }
  L.bytes = c.off;
  return L;
}

struct MlpBwdLayout {
  void *dz = nullptr, *dh1 = nullptr, *partials = nullptr;
  float* colsum = nullptr;
  size_t bytes = 0;
};

MlpBwdLayout mlp_bwd_layout(const tp_mlp_desc* d, void* scratch) {
  MlpBwdLayout L;
  Carver c(scratch);
  const size_t es = elem_size(d->dtype);
  const int64_t fp = d->act == TP_SWIGLU ? 2 * d->h_ffn : d->h_ffn;
  if (d->dropout_p > 0.0f) L.dz = c.take((size_t)d->T * (size_t)d->h * es);
  L.dh1 = c.take((size_t)d->T * (size_t)fp * es);
  if (d->mode != TP_REDUCE_FUSED)
    L.partials = c.take((size_t)d->n * (size_t)d->T * (size_t)d->h * es);
  L.colsum = static_cast<float*>(c.take(std::max(
      colsum_scratch_bytes(d->T, fp), colsum_scratch_bytes(d->T, d->h))));
  L.bytes = c.off;
  return L;
}

int reduce_d(int32_t dtype, const void* P, int n, int64_t rows, int64_t h,
             int64_t zstride, int64_t row0, const void* bias,
             const void* resid, void* out, const DropoutSpec& dr,
             tp_stream s) {
  return dtype == TP_F32
             ? reduce_partials<float>(P, n, rows, h, zstride, row0, bias,
                                      resid, out, dr, s)
             : reduce_partials<__nv_bfloat16>(P, n, rows, h, zstride, row0,
                                              bias, resid, out, dr, s);
}

// A second stream per device for the overlapped reductions, with a few
// events; one caller at a time enqueues through it.
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t ev[8] = {};
};
std::mutex g_side_mu;
SideStream g_side[64];

int side_stream(SideStream** out) {
  int dev = 0;
  int err = cudaGetDevice(&dev);
  if (err) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  SideStream& ss = g_side[dev];
  if (ss.s == nullptr) {
    err = cudaStreamCreateWithFlags(&ss.s, cudaStreamNonBlocking);
    for (int i = 0; !err && i < 8; ++i)
      err = cudaEventCreateWithFlags(&ss.ev[i], cudaEventDisableTiming);
    if (err) return err;
  }
  *out = &ss;
  return 0;
}

// A row-parallel projection (or input gradient) whose GEMM writes the n
// shard partials [n][T, h] (batch z = shard z), followed by their sum
// (+ bias, dropout, residual).  TP_REDUCE_MATERIALISED: the GEMM, then the
// reduce.  TP_REDUCE_OVERLAP: the rows are cut into bands ([Troverld]
// §II.II: the reduction of a tile can start as soon as the tile is
// computed); band b's GEMM runs on `stream`, then its reduce on a second
// stream after an event, while band b+1's GEMM runs; `stream` waits for the
// last reduce.  The arithmetic of every element is the same in both modes.
// The A operands of g are K-major [T, K] row blocks.
int gemm_and_reduce(const GemmProblem& g, int32_t sdt, void* partials, int n,
                    int64_t T, int64_t h, const void* bias, const void* resid,
                    void* out, const DropoutSpec& dr, int32_t mode,
                    tp_stream stream) {
  const size_t eo = elem_size(sdt);
  if (mode != TP_REDUCE_OVERLAP || T < 2048) {
    int err = run_gemm(g, stream);
    if (err) return err;
    return reduce_d(sdt, partials, n, T, h, T * h, 0, bias, resid, out, dr,
                    stream);
  }
  const size_t ea = g.dtype == TP_FP8 ? 1 : eo;
  const int nb = (int)std::min<int64_t>(4, T / 1024);
  // bands of whole 256-row pair tiles
  const int64_t band = (T / nb + 255) / 256 * 256;
  std::lock_guard<std::mutex> lk(g_side_mu);
  SideStream* ss = nullptr;
  int err = side_stream(&ss);
  if (err) return err;
  cudaStream_t main_s = static_cast<cudaStream_t>(stream);
  int b = 0;
  for (int64_t r0 = 0; r0 < T; r0 += band, ++b) {
    const int64_t rows = std::min(band, T - r0);
    GemmProblem gb = g;
    gb.M = rows;
    for (int p = 0; p < g.nparts; ++p) {
      gb.parts[p].a.ptr = static_cast<const char*>(g.parts[p].a.ptr) +
                          (size_t)r0 * (size_t)g.parts[p].a.ld * ea;
      gb.parts[p].a.rows = rows;
    }
    gb.epi.out = static_cast<char*>(partials) + (size_t)r0 * (size_t)h * eo;
    err = run_gemm(gb, stream);
    if (!err) err = cudaEventRecord(ss->ev[b], main_s);
    if (!err) err = cudaStreamWaitEvent(ss->s, ss->ev[b], 0);
    if (!err)
      err = reduce_d(sdt, static_cast<char*>(partials) + (size_t)r0 * h * eo,
                     n, rows, h, T * h, r0, bias,
                     resid ? static_cast<const char*>(resid) + r0 * h * eo
                           : nullptr,
                     static_cast<char*>(out) + (size_t)r0 * h * eo, dr, ss->s);
    if (err) return err;
  }
  err = cudaEventRecord(ss->ev[b], ss->s);
  if (!err) err = cudaStreamWaitEvent(main_s, ss->ev[b], 0);
  return err;
}

int colsum_d(int32_t dtype, const void* X, int64_t rows, int64_t cols,
             void* out, float* scratch, tp_stream s) {
  return dtype == TP_F32
             ? colsum<float>(X, rows, cols, cols, out, scratch, s)
             : colsum<__nv_bfloat16>(X, rows, cols, cols, out, scratch, s);
}

GemmOperand op(const void* p, int64_t ld, int mn, int64_t rows) {
  GemmOperand o;
  o.ptr = p;
  o.ld = ld;
  o.mn_major = mn;
  o.rows = rows;
  return o;
}

}  // namespace

extern "C" size_t tp_mlp_workspace_bytes(const tp_mlp_desc* d) {
  if (check_mlp(d) != TP_OK) return 0;
  return mlp_fwd_layout(d, nullptr).bytes;
}

extern "C" size_t tp_mlp_bwd_scratch_bytes(const tp_mlp_desc* d) {
  if (check_mlp(d) != TP_OK) return 0;
  return mlp_bwd_layout(d, nullptr).bytes;
}

extern "C" tp_status tp_mlp_fwd(const tp_mlp_desc* d, const void* X,
                                const void* W1, const void* b1, const void* W2,
                                const void* b2, const void* R, void* Out,
                                void* ws, size_t ws_bytes, tp_stream stream) {
  return guarded([&]() -> tp_status {
    tp_status st = check_mlp(d);
    if (st != TP_OK) return st;
    if (!X || !W1 || !W2 || !Out || !ws) return TP_ERR_NULL;
    if (!aligned16(X) || !aligned16(W1) || !aligned16(W2) || !aligned16(Out) ||
        !aligned16(ws) || !opt_aligned(b1) || !opt_aligned(b2) ||
        !opt_aligned(R))
      return TP_ERR_ARG;
    if (d->act == TP_SWIGLU && b1 != nullptr) return TP_ERR_UNSUPPORTED;
    const MlpFwdLayout L = mlp_fwd_layout(d, ws);
    if (ws_bytes < L.bytes) return TP_ERR_WORKSPACE;
    const int64_t T = d->T, h = d->h, f = d->h_ffn;
    const int n = d->n;
    const size_t es = elem_size(d->dtype);
    const DropoutSpec dr = make_dropout(d->dropout_p, d->seed);

    const bool f8 = d->dtype == TP_FP8;
    int err = 0;
    if (f8) {   // quantize the first projection's operands
      const int64_t w1rows = d->act == TP_SWIGLU ? 2 * f : f;
      err = quantize_fp8(X, T * h, L.xq, L.scales + 0, L.amax + 0, stream);
      if (!err)
        err = quantize_fp8(W1, w1rows * h, L.w1q, L.scales + 1, L.amax + 1,
                           stream);
      if (err) return cuda_status(err);
    }

    // column-parallel first projection + activation (shard-local)
    GemmProblem g1;
    g1.dtype = d->dtype;
    g1.M = T;
    g1.N = f;
    g1.parts[0].a = op(f8 ? L.xq : X, h, 0, T);
    g1.parts[0].b = op(f8 ? L.w1q : W1, h, 0, f);
    g1.parts[0].kseg = h;
    if (f8) {
      g1.epi.scale_a = L.scales + 0;
      g1.epi.scale_b = L.scales + 1;
    }
    if (d->act == TP_GELU) {
      g1.epi.kind = EPI_GELU;
      g1.epi.out = L.h_or_g;
      g1.epi.out2 = L.a;
      g1.epi.bias = b1;
    } else {
      g1.parts[0].b2 =
          f8 ? op(static_cast<const char*>(L.w1q) + (size_t)f * h, h, 0, f)
             : op(static_cast<const char*>(W1) + (size_t)f * h * es, h, 0, f);
      g1.epi.kind = EPI_SWIGLU;
      g1.epi.out = L.h_or_g;
      g1.epi.out2 = L.u;
      g1.epi.out3 = L.a;
    }
    g1.epi.ldo = f;
    g1.epi.ldo2 = f;
    err = run_gemm(g1, stream);
    if (err) return cuda_status(err);
    if (f8) {   // quantize the second projection's operands
      err = quantize_fp8(L.a, T * f, L.aq, L.scales + 2, L.amax + 2, stream);
      if (!err)
        err = quantize_fp8(W2, h * f, L.w2q, L.scales + 3, L.amax + 3, stream);
      if (err) return cuda_status(err);
    }

    // row-parallel second projection + g reduction + bias/dropout/residual
    GemmProblem g2;
    g2.dtype = d->dtype;
    g2.M = T;
    g2.N = h;
    g2.parts[0].a = op(f8 ? L.aq : L.a, f, 0, T);
    g2.parts[0].b = op(f8 ? L.w2q : W2, f, 0, h);
    if (f8) {
      g2.epi.scale_a = L.scales + 2;
      g2.epi.scale_b = L.scales + 3;
    }
    if (d->mode == TP_REDUCE_FUSED) {
      g2.parts[0].kseg = f;
      g2.epi.kind = EPI_STORE;
      g2.epi.out = Out;
      g2.epi.ldo = h;
      g2.epi.bias = b2;
      g2.epi.resid = R;
      g2.epi.ldr = h;
      g2.epi.dropout = dr.enabled;
      g2.epi.drop_thr = dr.thr;
      g2.epi.drop_scale = dr.scale;
      g2.epi.seed = dr.seed;
      return cuda_status(run_gemm(g2, stream));
    }
    g2.parts[0].kseg = f / n;
    g2.parts[0].nseg = n;
    g2.parts[0].seg_z_stride = 1;
    g2.nz = n;
    g2.epi.kind = EPI_STORE;
    g2.epi.out = L.partials;
    g2.epi.ldo = h;
    g2.epi.out_z_stride = T * h;
    return cuda_status(gemm_and_reduce(g2, storage(d->dtype), L.partials, n,
                                       T, h, b2, R, Out, dr, d->mode, stream));
  });
}

namespace {
// leave_partials (non-fused modes): the f reduction's shard partials of dX
// are left in the scratch and their address reported to the caller; dX and
// dres are not touched.
tp_status mlp_bwd_impl(const tp_mlp_desc* d, const void* dOut, const void* X,
                       const void* W1, const void* W2, const void* ws,
                       const void* dres, void* dX, void* dW1, void* db1,
                       void* dW2, void* db2, void* scratch,
                       size_t scratch_bytes, tp_stream stream,
                       void** leave_partials);
}  // namespace

extern "C" tp_status tp_mlp_bwd(const tp_mlp_desc* d, const void* dOut,
                                const void* X, const void* W1, const void* W2,
                                const void* ws, const void* dres, void* dX,
                                void* dW1, void* db1, void* dW2, void* db2,
                                void* scratch, size_t scratch_bytes,
                                tp_stream stream) {
  return mlp_bwd_impl(d, dOut, X, W1, W2, ws, dres, dX, dW1, db1, dW2, db2,
                      scratch, scratch_bytes, stream, nullptr);
}

namespace {
tp_status mlp_bwd_impl(const tp_mlp_desc* d, const void* dOut, const void* X,
                       const void* W1, const void* W2, const void* ws,
                       const void* dres, void* dX, void* dW1, void* db1,
                       void* dW2, void* db2, void* scratch,
                       size_t scratch_bytes, tp_stream stream,
                       void** leave_partials) {
  return guarded([&]() -> tp_status {
    tp_status st = check_mlp(d);
    if (st != TP_OK) return st;
    const int32_t sdt = storage(d->dtype);   // FP8 mode: bf16 backward
    if (!dOut || !X || !W1 || !W2 || !ws || !dX || !dW1 || !dW2 || !scratch)
      return TP_ERR_NULL;
    if (!aligned16(dOut) || !aligned16(X) || !aligned16(W1) ||
        !aligned16(W2) || !aligned16(ws) || !aligned16(dX) ||
        !aligned16(dW1) || !aligned16(dW2) || !aligned16(scratch) ||
        !opt_aligned(dres) || !opt_aligned(db1) || !opt_aligned(db2))
      return TP_ERR_ARG;
    const MlpFwdLayout F = mlp_fwd_layout(d, const_cast<void*>(ws));
    const MlpBwdLayout L = mlp_bwd_layout(d, scratch);
    if (scratch_bytes < L.bytes) return TP_ERR_WORKSPACE;
    const int64_t T = d->T, h = d->h, f = d->h_ffn;
    const int n = d->n;
    const bool swiglu = d->act == TP_SWIGLU;
    const int64_t fp = swiglu ? 2 * f : f;
    const size_t es = elem_size(sdt);
    const DropoutSpec dr = make_dropout(d->dropout_p, d->seed);
    int err = 0;

    // dZ = dOut ⊙ mask/(1−p)
    const void* dZ = dOut;
    if (dr.enabled) {
      err = sdt == TP_F32
                ? dropout_bwd<float>(dOut, T * h, L.dz, dr, stream)
                : dropout_bwd<__nv_bfloat16>(dOut, T * h, L.dz, dr, stream);
      if (err) return cuda_status(err);
      dZ = L.dz;
    }
    if (db2) {
      err = colsum_d(sdt, dZ, T, h, db2, L.colsum, stream);
      if (err) return cuda_status(err);
    }
    // dA = dZ·W2 (shard-local columns), through the activation
    GemmProblem ga;
    ga.dtype = sdt;
    ga.M = T;
    ga.N = f;
    ga.parts[0].a = op(dZ, h, 0, T);
    ga.parts[0].b = op(W2, f, 1, f);
    ga.parts[0].kseg = h;
    if (!swiglu) {
      ga.epi.kind = EPI_DGELU;
      ga.epi.out = L.dh1;
      ga.epi.ldo = f;
      ga.epi.aux1 = F.h_or_g;
      ga.epi.ld_aux = f;
    } else {
      ga.epi.kind = EPI_DSWIGLU;
      ga.epi.out = L.dh1;
      ga.epi.out2 = static_cast<char*>(L.dh1) + (size_t)f * es;
      ga.epi.ldo = 2 * f;
      ga.epi.aux1 = F.h_or_g;
      ga.epi.aux2 = F.u;
      ga.epi.ld_aux = f;
    }
    err = run_gemm(ga, stream);
    if (err) return cuda_status(err);
    if (db1) {
      err = colsum_d(sdt, L.dh1, T, fp, db1, L.colsum, stream);
      if (err) return cuda_status(err);
    }
    // dW2 = dZᵀ·A  [h, f]
    GemmProblem gw2;
    gw2.dtype = sdt;
    gw2.M = h;
    gw2.N = f;
    gw2.parts[0].a = op(dZ, h, 1, h);
    gw2.parts[0].b = op(F.a, f, 1, f);
    gw2.parts[0].kseg = T;
    gw2.epi.kind = EPI_STORE;
    gw2.epi.out = dW2;
    gw2.epi.ldo = f;
    err = run_gemm(gw2, stream);
    if (err) return cuda_status(err);
    // dW1 = dH1ᵀ·X  [fp, h]
    GemmProblem gw1;
    gw1.dtype = sdt;
    gw1.M = fp;
    gw1.N = h;
    gw1.parts[0].a = op(L.dh1, fp, 1, fp);
    gw1.parts[0].b = op(X, h, 1, h);
    gw1.parts[0].kseg = T;
    gw1.epi.kind = EPI_STORE;
    gw1.epi.out = dW1;
    gw1.epi.ldo = h;
    err = run_gemm(gw1, stream);
    if (err) return cuda_status(err);
    // f: dX = Σ_i dH1_i·W1_i (+ dres)
    GemmProblem gx;
    gx.dtype = sdt;
    gx.M = T;
    gx.N = h;
    gx.parts[0].a = op(L.dh1, fp, 0, T);
    gx.parts[0].b = op(W1, h, 1, h);
    gx.epi.kind = EPI_STORE;
    gx.epi.ldo = h;
    if (d->mode == TP_REDUCE_FUSED) {
      gx.parts[0].kseg = fp;
      gx.epi.out = dX;
      gx.epi.resid = dres;
      gx.epi.ldr = h;
      return cuda_status(run_gemm(gx, stream));
    }
    const int64_t w = f / n;
    gx.parts[0].kseg = w;
    gx.parts[0].nseg = (int)(fp / w);
    gx.parts[0].seg_z_stride = 1;
    gx.parts[0].nsub = swiglu ? 2 : 1;
    gx.parts[0].seg_sub_stride = n;
    gx.nz = n;
    gx.epi.out = L.partials;
    gx.epi.out_z_stride = T * h;
    if (leave_partials) {
      *leave_partials = L.partials;
      return cuda_status(run_gemm(gx, stream));
    }
    return cuda_status(gemm_and_reduce(gx, sdt, L.partials, n, T, h, nullptr,
                                       dres, dX, DropoutSpec(), d->mode,
                                       stream));
  });
}
}  // namespace

// ------------------------------------------------------------- attention --
namespace {

tp_status check_attn(const tp_attn_desc* d) {
  if (d == nullptr) return TP_ERR_NULL;
  if (d->dtype != TP_F32 && d->dtype != TP_BF16 && d->dtype != TP_FP8)
    return TP_ERR_DTYPE;
  if (d->mode != TP_REDUCE_FUSED && d->mode != TP_REDUCE_MATERIALISED &&
      d->mode != TP_REDUCE_OVERLAP && d->mode != TP_REDUCE_SP)
    return TP_ERR_DTYPE;
  if (d->b < 1 || d->s < 1 || d->h < 8 || d->n_q < 1 || d->n_kv < 1 ||
      d->d < 1 || d->n < 1)
    return TP_ERR_SHAPE;
  if (d->b * d->s > (1 << 30) || d->h > (1 << 20) || d->h % 8)
    return TP_ERR_SHAPE;
  // GQA groups and heads must split evenly over the n ranks
  if (d->n_q % d->n_kv || d->n_q % d->n || d->n_kv % d->n) return TP_ERR_SHAPE;
  if (storage(d->dtype) != TP_BF16 || d->d != 128) return TP_ERR_UNSUPPORTED;
  // FP8 mode: E4M3 rows of X (h bytes) must start on 16-byte boundaries
  if (d->dtype == TP_FP8 && d->h % 16) return TP_ERR_SHAPE;
  return TP_OK;
}

struct AttnFwdLayout {
  void *q = nullptr, *k = nullptr, *v = nullptr, *o = nullptr;
  float* lse = nullptr;
  void* partials = nullptr;
  // FP8 mode: E4M3 copies of X, Wq, Wk, Wv, O, Wo, their scales (same
  // order) and amax scratch words
  void *xq = nullptr, *wqq = nullptr, *wkq = nullptr, *wvq = nullptr,
       *oq = nullptr, *woq = nullptr;
  float* scales = nullptr;
  unsigned* amax = nullptr;
  size_t bytes = 0;
};

AttnFwdLayout attn_fwd_layout(const tp_attn_desc* d, void* ws) {
  AttnFwdLayout L;
  Carver c(ws);
  const size_t T = (size_t)d->b * (size_t)d->s;
  const size_t qd = (size_t)d->n_q * d->d, kd = (size_t)d->n_kv * d->d;
  L.q = c.take(T * qd * 2);
  L.k = c.take(T * kd * 2);
  L.v = c.take(T * kd * 2);
  L.o = c.take(T * qd * 2);
  L.lse = static_cast<float*>(c.take((size_t)d->b * d->n_q * d->s * 4));
  if (d->mode != TP_REDUCE_FUSED)
    L.partials = c.take((size_t)d->n * T * (size_t)d->h * 2);
  if (d->dtype == TP_FP8) {
    const size_t h = (size_t)d->h;
    L.xq = c.take(T * h);
    L.wqq = c.take(qd * h);
    L.wkq = c.take(kd * h);
    L.wvq = c.take(kd * h);
    L.oq = c.take(T * qd);
    L.woq = c.take(h * qd);
    L.scales = static_cast<float*>(c.take(6 * sizeof(float)));
    L.amax = static_cast<unsigned*>(c.take(6 * sizeof(unsigned)));
  }
  L.bytes = c.off;
  return L;
}

struct AttnBwdLayout {
  void *dO = nullptr, *dQ = nullptr, *dK = nullptr, *dV = nullptr;
  void* dS = nullptr;
  float *D = nullptr, *L2 = nullptr;
  void* partials = nullptr;
  float* colsum = nullptr;
  size_t bytes = 0;
};

AttnShape attn_shape(const tp_attn_desc* d);

// `sh` carries the dS pairs per pass, fixed once per call (attn_shape).
AttnBwdLayout attn_bwd_layout(const tp_attn_desc* d, const AttnShape& sh,
                              void* scratch) {
  AttnBwdLayout L;
  Carver c(scratch);
  const size_t T = (size_t)d->b * (size_t)d->s;
  const size_t qd = (size_t)d->n_q * d->d, kd = (size_t)d->n_kv * d->d;
  L.dO = c.take(T * qd * 2);
  L.dQ = c.take(T * qd * 2);
  L.dK = c.take(T * kd * 2);
  L.dV = c.take(T * kd * 2);
  const size_t stats = (size_t)d->b * d->n_q * attn_stats_pad(d->s) * 4;
  L.D = static_cast<float*>(c.take(stats));
  L.L2 = static_cast<float*>(c.take(stats));
  L.dS = c.take((size_t)attn_ds_bytes(sh));
  if (d->mode != TP_REDUCE_FUSED)
    L.partials = c.take((size_t)d->n * T * (size_t)d->h * 2);
  L.colsum = static_cast<float*>(c.take(colsum_scratch_bytes(T, d->h)));
  L.bytes = c.off;
  return L;
}

AttnShape attn_shape(const tp_attn_desc* d) {
  AttnShape sh;
  sh.b = d->b;
  sh.s = d->s;
  sh.nq = d->n_q;
  sh.nkv = d->n_kv;
  sh.d = d->d;
  sh.causal = d->causal ? 1 : 0;
  sh.scale = 1.0f / std::sqrt((float)d->d);
  sh.ds_pairs = attn_ds_pairs_per_pass(sh);   // the one read of the budget
  return sh;
}

GemmProblem proj(int64_t M, int64_t N, const GemmOperand& a,
                 const GemmOperand& b, int64_t K, void* out, int64_t ldo) {
  GemmProblem g;
  g.dtype = TP_BF16;
  g.M = M;
  g.N = N;
  g.parts[0].a = a;
  g.parts[0].b = b;
  g.parts[0].kseg = K;
  g.epi.kind = EPI_STORE;
  g.epi.out = out;
  g.epi.ldo = ldo;
  return g;
}

}  // namespace

extern "C" size_t tp_attn_workspace_bytes(const tp_attn_desc* d) {
  if (check_attn(d) != TP_OK) return 0;
  return attn_fwd_layout(d, nullptr).bytes;
}

extern "C" size_t tp_attn_bwd_scratch_bytes(const tp_attn_desc* d) {
  if (check_attn(d) != TP_OK) return 0;
  return attn_bwd_layout(d, attn_shape(d), nullptr).bytes;
}

namespace {
// fp16 copies of the Q, K, V projections' operands: the input rows and the
// three weights, stacked [Wq; Wk; Wv] so that one launch computes all three
// projections.  The layer passes them for its first block, whose input is
// the RMSNorm output: the softmax amplifies the rounding of that input
// (scores of a few units times its relative error), and fp16 keeps 3 more
// mantissa bits than bf16 at the same bytes.
struct QkvF16 {
  const void *x = nullptr, *wqkv = nullptr;
};

tp_status attn_fwd_impl(const tp_attn_desc* d, const void* X, const void* Wq,
                        const void* Wk, const void* Wv, const void* Wo,
                        const void* bo, const void* R, void* Out, void* ws,
                        size_t ws_bytes, tp_stream stream,
                        const QkvF16* f16in, void** leave_partials = nullptr);
}  // namespace

extern "C" tp_status tp_attn_fwd(const tp_attn_desc* d, const void* X,
                                 const void* Wq, const void* Wk,
                                 const void* Wv, const void* Wo,
                                 const void* bo, const void* R, void* Out,
                                 void* ws, size_t ws_bytes, tp_stream stream) {
  return attn_fwd_impl(d, X, Wq, Wk, Wv, Wo, bo, R, Out, ws, ws_bytes, stream,
                       nullptr);
}

namespace {
// leave_partials (non-fused modes): stop after the output projection's
// shard partials are written and report where they are (the caller reduces
// them).
tp_status attn_fwd_impl(const tp_attn_desc* d, const void* X, const void* Wq,
                        const void* Wk, const void* Wv, const void* Wo,
                        const void* bo, const void* R, void* Out, void* ws,
                        size_t ws_bytes, tp_stream stream,
                        const QkvF16* f16in, void** leave_partials) {
  return guarded([&]() -> tp_status {
    tp_status st = check_attn(d);
    if (st != TP_OK) return st;
    if (!X || !Wq || !Wk || !Wv || !Wo || !Out || !ws) return TP_ERR_NULL;
    if (!aligned16(X) || !aligned16(Wq) || !aligned16(Wk) || !aligned16(Wv) ||
        !aligned16(Wo) || !aligned16(Out) || !aligned16(ws) ||
        !opt_aligned(bo) || !opt_aligned(R))
      return TP_ERR_ARG;
    const AttnFwdLayout L = attn_fwd_layout(d, ws);
    if (ws_bytes < L.bytes) return TP_ERR_WORKSPACE;
    const int64_t T = d->b * d->s, h = d->h;
    const int64_t qd = (int64_t)d->n_q * d->d, kd = (int64_t)d->n_kv * d->d;
    const int n = d->n;
    const bool f8 = d->dtype == TP_FP8;
    int err = 0;
    if (f8) {   // quantize the projections' operands, one scale per tensor
      const void* src[4] = {X, Wq, Wk, Wv};
      void* dst[4] = {L.xq, L.wqq, L.wkq, L.wvq};
      const int64_t cnt[4] = {T * h, qd * h, kd * h, kd * h};
      for (int i = 0; i < 4 && !err; ++i)
        err = quantize_fp8(src[i], cnt[i], dst[i], L.scales + i, L.amax + i,
                           stream);
      if (err) return cuda_status(err);
    }
    // column-parallel Q, K, V projections (each rank's heads are a column
    // block, written in fp16 for the attention core)
    const void* xa = f8 ? L.xq : X;
    GemmProblem gq = proj(T, qd, op(xa, h, 0, T), op(f8 ? L.wqq : Wq, h, 0, qd),
                          h, L.q, qd);
    GemmProblem gk = proj(T, kd, op(xa, h, 0, T), op(f8 ? L.wkq : Wk, h, 0, kd),
                          h, L.k, kd);
    GemmProblem gv = proj(T, kd, op(xa, h, 0, T), op(f8 ? L.wvq : Wv, h, 0, kd),
                          h, L.v, kd);
    gq.epi.out_f16 = gk.epi.out_f16 = gv.epi.out_f16 = 1;
    const bool fused_qkv = f16in != nullptr && !f8;
    if (fused_qkv) {
      // one launch over the stacked fp16 weights: columns [0, qd) are Q,
      // [qd, qd + kd) K and the rest V (tile widths divide qd and kd)
      gq = proj(T, qd + 2 * kd, op(f16in->x, h, 0, T),
                op(f16in->wqkv, h, 0, qd + 2 * kd), h, L.q, qd);
      gq.f16 = 1;
      gq.epi.out_f16 = 1;
      gq.epi.split1 = qd;
      gq.epi.out2 = L.k;
      gq.epi.ldo2 = kd;
      gq.epi.split2 = qd + kd;
      gq.epi.out3 = L.v;
      gq.epi.ldo3 = kd;
    }
    if (f8) {
      GemmProblem* gs[3] = {&gq, &gk, &gv};
      for (int i = 0; i < 3; ++i) {
        gs[i]->dtype = TP_FP8;
        gs[i]->epi.scale_a = L.scales + 0;
        gs[i]->epi.scale_b = L.scales + 1 + i;
      }
    }
    err = run_gemm(gq, stream);
    if (!err && !fused_qkv) err = run_gemm(gk, stream);
    if (!err && !fused_qkv) err = run_gemm(gv, stream);
    if (err) return cuda_status(err);
    err = flash_fwd(attn_shape(d), L.q, L.k, L.v, L.o, L.lse,
                    device_status_ptr(), stream);
    if (err) return cuda_status(err);
    if (f8) {   // O (bf16) and Wo to E4M3
      err = quantize_fp8(L.o, T * qd, L.oq, L.scales + 4, L.amax + 4, stream);
      if (!err)
        err = quantize_fp8(Wo, h * qd, L.woq, L.scales + 5, L.amax + 5,
                           stream);
      if (err) return cuda_status(err);
    }
    // row-parallel output projection + g reduction + bias + residual
    GemmProblem g = proj(T, h, op(f8 ? L.oq : L.o, qd, 0, T),
                         op(f8 ? L.woq : Wo, qd, 0, h), qd, Out, h);
    if (f8) {
      g.dtype = TP_FP8;
      g.epi.scale_a = L.scales + 4;
      g.epi.scale_b = L.scales + 5;
    }
    if (d->mode == TP_REDUCE_FUSED) {
      g.epi.bias = bo;
      g.epi.resid = R;
      g.epi.ldr = h;
      return cuda_status(run_gemm(g, stream));
    }
    g.parts[0].kseg = qd / n;
    g.parts[0].nseg = n;
    g.parts[0].seg_z_stride = 1;
    g.nz = n;
    g.epi.out = L.partials;
    g.epi.out_z_stride = T * h;
    if (leave_partials) {
      *leave_partials = L.partials;
      return cuda_status(run_gemm(g, stream));
    }
    return cuda_status(gemm_and_reduce(g, TP_BF16, L.partials, n, T, h, bo, R,
                                       Out, DropoutSpec(), d->mode, stream));
  });
}

}  // namespace

namespace {
// leave_partials (non-fused modes): the f reduction's shard partials of dX
// are left in the scratch and their address reported to the caller; dX and
// dres are not touched.
tp_status attn_bwd_impl(const tp_attn_desc* d, const void* dOut,
                        const void* X, const void* Wq, const void* Wk,
                        const void* Wv, const void* Wo, const void* ws,
                        const void* dres, void* dX, void* dWq, void* dWk,
                        void* dWv, void* dWo, void* dbo, void* scratch,
                        size_t scratch_bytes, tp_stream stream,
                        void** leave_partials);
}  // namespace

extern "C" tp_status tp_attn_bwd(const tp_attn_desc* d, const void* dOut,
                                 const void* X, const void* Wq, const void* Wk,
                                 const void* Wv, const void* Wo,
                                 const void* ws, const void* dres, void* dX,
                                 void* dWq, void* dWk, void* dWv, void* dWo,
                                 void* dbo, void* scratch,
                                 size_t scratch_bytes, tp_stream stream) {
  return attn_bwd_impl(d, dOut, X, Wq, Wk, Wv, Wo, ws, dres, dX, dWq, dWk,
                       dWv, dWo, dbo, scratch, scratch_bytes, stream, nullptr);
}

namespace {
tp_status attn_bwd_impl(const tp_attn_desc* d, const void* dOut,
                        const void* X, const void* Wq, const void* Wk,
                        const void* Wv, const void* Wo, const void* ws,
                        const void* dres, void* dX, void* dWq, void* dWk,
                        void* dWv, void* dWo, void* dbo, void* scratch,
                        size_t scratch_bytes, tp_stream stream,
                        void** leave_partials) {
  return guarded([&]() -> tp_status {
    tp_status st = check_attn(d);
    if (st != TP_OK) return st;
    if (!dOut || !X || !Wq || !Wk || !Wv || !Wo || !ws || !dX || !dWq ||
        !dWk || !dWv || !dWo || !scratch)
      return TP_ERR_NULL;
    if (!aligned16(dOut) || !aligned16(X) || !aligned16(Wq) ||
        !aligned16(Wk) || !aligned16(Wv) || !aligned16(Wo) || !aligned16(ws) ||
        !aligned16(dX) || !aligned16(dWq) || !aligned16(dWk) ||
        !aligned16(dWv) || !aligned16(dWo) || !aligned16(scratch) ||
        !opt_aligned(dres) || !opt_aligned(dbo))
      return TP_ERR_ARG;
    const AttnFwdLayout F = attn_fwd_layout(d, const_cast<void*>(ws));
    // one shape (and one read of the dS budget) for the layout and the
    // kernels, so the tiles written always fit the carved region
    const AttnShape sh = attn_shape(d);
    const AttnBwdLayout L = attn_bwd_layout(d, sh, scratch);
    if (scratch_bytes < L.bytes) return TP_ERR_WORKSPACE;
    const int64_t T = d->b * d->s, h = d->h;
    const int64_t qd = (int64_t)d->n_q * d->d, kd = (int64_t)d->n_kv * d->d;
    const int n = d->n;
    int err = 0;
    if (dbo) {
      err = colsum<__nv_bfloat16>(dOut, T, h, h, dbo, L.colsum, stream);
      if (err) return cuda_status(err);
    }
    // dO = dOut·Wo (local), dWo = dOutᵀ·O
    GemmProblem gdo = proj(T, qd, op(dOut, h, 0, T), op(Wo, qd, 1, qd), h,
                           L.dO, qd);
    gdo.epi.out_f16 = 1;   // attention-core operand
    err = run_gemm(gdo, stream);
    if (!err)
      err = run_gemm(proj(h, qd, op(dOut, h, 1, h), op(F.o, qd, 1, qd), T, dWo,
                          qd),
                     stream);
    if (err) return cuda_status(err);
    err = flash_bwd(sh, F.q, F.k, F.v, F.o, L.dO, F.lse, L.D, L.L2,
                    L.dS, L.dQ, L.dK, L.dV, device_status_ptr(), stream);
    if (err) return cuda_status(err);
    err = run_gemm(proj(qd, h, op(L.dQ, qd, 1, qd), op(X, h, 1, h), T, dWq, h),
                   stream);
    if (!err)
      err = run_gemm(proj(kd, h, op(L.dK, kd, 1, kd), op(X, h, 1, h), T, dWk,
                          h),
                     stream);
    if (!err)
      err = run_gemm(proj(kd, h, op(L.dV, kd, 1, kd), op(X, h, 1, h), T, dWv,
                          h),
                     stream);
    if (err) return cuda_status(err);
    // f: dX = Σ_i (dQ_i Wq_i + dK_i Wk_i + dV_i Wv_i) (+ dres)
    GemmProblem g = proj(T, h, op(L.dQ, qd, 0, T), op(Wq, h, 1, h), qd, dX, h);
    g.nparts = 3;
    g.parts[1].a = op(L.dK, kd, 0, T);
    g.parts[1].b = op(Wk, h, 1, h);
    g.parts[1].kseg = kd;
    g.parts[2].a = op(L.dV, kd, 0, T);
    g.parts[2].b = op(Wv, h, 1, h);
    g.parts[2].kseg = kd;
    if (d->mode == TP_REDUCE_FUSED) {
      g.epi.resid = dres;
      g.epi.ldr = h;
      return cuda_status(run_gemm(g, stream));
    }
    g.parts[0].kseg = qd / n;
    g.parts[1].kseg = kd / n;
    g.parts[2].kseg = kd / n;
    for (int i = 0; i < 3; ++i) {
      g.parts[i].nseg = n;
      g.parts[i].seg_z_stride = 1;
    }
    g.nz = n;
    g.epi.out = L.partials;
    g.epi.out_z_stride = T * h;
    if (leave_partials) {
      *leave_partials = L.partials;
      return cuda_status(run_gemm(g, stream));
    }
    return cuda_status(gemm_and_reduce(g, TP_BF16, L.partials, n, T, h,
                                       nullptr, dres, dX, DropoutSpec(),
                                       d->mode, stream));
  });
}
}  // namespace

// -------------------------------------------------------------- RMSNorm --
extern "C" tp_status tp_rmsnorm_fwd(int64_t T, int64_t h, float eps,
                                    int32_t dtype, const void* x,
                                    const void* gamma, void* y, float* rstd,
                                    tp_stream stream) {
  return guarded([&]() -> tp_status {
    if (dtype != TP_F32 && dtype != TP_BF16) return TP_ERR_DTYPE;
    if (T < 1 || h < 8 || h % 8 || h > 16384) return TP_ERR_SHAPE;
    if (!x || !gamma || !y || !rstd) return TP_ERR_NULL;
    if (!aligned16(x) || !aligned16(gamma) || !aligned16(y) || !aligned16(rstd))
      return TP_ERR_ARG;
    const int err =
        dtype == TP_F32
            ? rmsnorm_fwd<float>(x, gamma, y, rstd, T, h, eps, stream)
            : rmsnorm_fwd<__nv_bfloat16>(x, gamma, y, rstd, T, h, eps, stream);
    return cuda_status(err);
  });
}

extern "C" size_t tp_rmsnorm_bwd_scratch_bytes(int64_t T, int64_t h) {
  if (T < 1 || h < 1) return 0;
  return rmsnorm_bwd_scratch(T, h);
}

extern "C" tp_status tp_rmsnorm_bwd(int64_t T, int64_t h, float eps,
                                    int32_t dtype, const void* dy,
                                    const void* x, const void* gamma,
                                    const float* rstd, const void* dres,
                                    void* dx, void* dgamma, void* scratch,
                                    size_t scratch_bytes, tp_stream stream) {
  (void)eps;  // rstd carries ε from the forward call
  return guarded([&]() -> tp_status {
    if (dtype != TP_F32 && dtype != TP_BF16) return TP_ERR_DTYPE;
    if (T < 1 || h < 8 || h % 8 || h > 16384) return TP_ERR_SHAPE;
    if (!dy || !x || !gamma || !rstd || !dx || !dgamma || !scratch)
      return TP_ERR_NULL;
    if (!aligned16(dy) || !aligned16(x) || !aligned16(gamma) ||
        !aligned16(rstd) || !aligned16(dx) || !opt_aligned(dres) ||
        !aligned16(scratch))
      return TP_ERR_ARG;
    if (scratch_bytes < rmsnorm_bwd_scratch(T, h)) return TP_ERR_WORKSPACE;
    float* sc = static_cast<float*>(scratch);
    const int err =
        dtype == TP_F32
            ? rmsnorm_bwd<float>(dy, x, gamma, rstd, dres, dx, dgamma, sc, T,
                                 h, stream)
            : rmsnorm_bwd<__nv_bfloat16>(dy, x, gamma, rstd, dres, dx, dgamma,
                                         sc, T, h, stream);
    return cuda_status(err);
  });
}

extern "C" tp_status tp_rmsnorm_bwd_noalloc(int64_t T, int64_t h, float eps,
                                            int32_t dtype, const void* dy,
                                            const void* x, const void* gamma,
                                            const float* rstd,
                                            const void* dres, void* dx,
                                            void* dgamma, tp_stream stream) {
  (void)eps;  // rstd carries ε from the forward call
  return guarded([&]() -> tp_status {
    if (dtype != TP_F32 && dtype != TP_BF16) return TP_ERR_DTYPE;
    if (T < 1 || h < 8 || h % 8 || h > 16384) return TP_ERR_SHAPE;
    if (h > TP_RMSNORM_NOALLOC_MAX_H) return TP_ERR_WORKSPACE;
    if (!dy || !x || !gamma || !rstd || !dx || !dgamma) return TP_ERR_NULL;
    if (!aligned16(dy) || !aligned16(x) || !aligned16(gamma) ||
        !aligned16(rstd) || !aligned16(dx) || !opt_aligned(dres))
      return TP_ERR_ARG;
    const int err =
        dtype == TP_F32
            ? rmsnorm_bwd_noalloc<float>(dy, x, gamma, rstd, dres, dx, dgamma,
                                         T, h, stream)
            : rmsnorm_bwd_noalloc<__nv_bfloat16>(dy, x, gamma, rstd, dres, dx,
                                                 dgamma, T, h, stream);
    return cuda_status(err);
  });
}

// ----------------------------------------------------------------- GEMM --
extern "C" tp_status tp_gemm(int32_t dtype, int64_t M, int64_t N, int64_t K,
                             const void* A, int64_t lda, int32_t a_mn_major,
                             const void* B, int64_t ldb, int32_t b_mn_major,
                             void* C, int64_t ldc, tp_stream stream) {
  return guarded([&]() -> tp_status {
    if (dtype != TP_F32 && dtype != TP_BF16) return TP_ERR_DTYPE;
    if (M < 1 || N < 1 || K < 1 || M > (1 << 30) || N > (1 << 30))
      return TP_ERR_SHAPE;
    if (!A || !B || !C) return TP_ERR_NULL;
    const int64_t q = dtype == TP_BF16 ? 8 : 4;
    if (lda % q || ldb % q || ldc % q || K % q) return TP_ERR_SHAPE;
    if (lda < (a_mn_major ? M : K) || ldb < (b_mn_major ? N : K) || ldc < N)
      return TP_ERR_SHAPE;
    if (!aligned16(A) || !aligned16(B) || !aligned16(C)) return TP_ERR_ARG;
    GemmProblem g;
    g.dtype = dtype;
    g.M = M;
    g.N = N;
    g.parts[0].a = op(A, lda, a_mn_major ? 1 : 0, M);
    g.parts[0].b = op(B, ldb, b_mn_major ? 1 : 0, N);
    g.parts[0].kseg = K;
    g.epi.kind = EPI_STORE;
    g.epi.out = C;
    g.epi.ldo = ldc;
    return cuda_status(run_gemm(g, stream));
  });
}

extern "C" tp_status tp_quantize_fp8(int64_t n, const void* x, void* q,
                                     float* scale_out, void* amax_work,
                                     tp_stream stream) {
  return guarded([&]() -> tp_status {
    if (!x || !q || !scale_out || !amax_work) return TP_ERR_NULL;
    if (n < 1 || n % 8) return TP_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(q) ||
        (reinterpret_cast<uintptr_t>(scale_out) & 3u) ||
        (reinterpret_cast<uintptr_t>(amax_work) & 3u))
      return TP_ERR_ARG;
    return cuda_status(quantize_fp8(x, n, q, scale_out,
                                    static_cast<unsigned*>(amax_work),
                                    stream));
  });
}

extern "C" tp_status tp_gemm_fp8(int64_t M, int64_t N, int64_t K,
                                 const void* qa, int64_t lda,
                                 const float* scale_a, const void* qb,
                                 int64_t ldb, const float* scale_b, void* C,
                                 int64_t ldc, tp_stream stream) {
  return guarded([&]() -> tp_status {
    if (!qa || !qb || !C || !scale_a || !scale_b) return TP_ERR_NULL;
    if (M < 1 || N < 1 || K < 1 || M > (1 << 30) || N > (1 << 30))
      return TP_ERR_SHAPE;
    if (lda % 16 || ldb % 16 || K % 16 || ldc % 8 || lda < K || ldb < K ||
        ldc < N)
      return TP_ERR_SHAPE;
    if (!aligned16(qa) || !aligned16(qb) || !aligned16(C)) return TP_ERR_ARG;
    GemmProblem g;
    g.dtype = TP_FP8;
    g.M = M;
    g.N = N;
    g.parts[0].a = op(qa, lda, 0, M);
    g.parts[0].b = op(qb, ldb, 0, N);
    g.parts[0].kseg = K;
    g.epi.kind = EPI_STORE;
    g.epi.out = C;
    g.epi.ldo = ldc;
    g.epi.scale_a = scale_a;
    g.epi.scale_b = scale_b;
    return cuda_status(run_gemm(g, stream));
  });
}

// ------------------------------------------------------------- profiling --
extern "C" tp_status tp_profile_enable(int32_t max_launches) {
  return guarded([&]() -> tp_status {
    std::lock_guard<std::mutex> lk(g_prof.mu);
    for (cudaEvent_t e : g_prof.ev)
      if (e != nullptr) cudaEventDestroy(e);
    g_prof.ev.clear();
    g_prof.rec.clear();
    g_prof.enabled = false;
    g_prof.max = g_prof.used = 0;
    if (max_launches <= 0) return TP_OK;
    g_prof.ev.resize(2 * (size_t)max_launches, nullptr);
    for (auto& e : g_prof.ev)
      if (cudaEventCreate(&e) != cudaSuccess) return TP_ERR_CUDA;
    g_prof.rec.resize((size_t)max_launches);
    g_prof.max = max_launches;
    g_prof.enabled = true;
    return TP_OK;
  });
}

extern "C" tp_status tp_profile_reset(void) {
  std::lock_guard<std::mutex> lk(g_prof.mu);
  g_prof.used = 0;
  return TP_OK;
}

extern "C" tp_status tp_profile_read(int32_t family, tp_profile_entry* out) {
  if (out == nullptr) return TP_ERR_NULL;
  if (family < 0 || family >= KF_COUNT) return TP_ERR_ARG;
  std::lock_guard<std::mutex> lk(g_prof.mu);
  tp_profile_entry r = {0, 0.0, 0.0, 0.0};
  for (int i = 0; i < g_prof.used; ++i) {
    if (g_prof.rec[i].family != family) continue;
    if (cudaEventSynchronize(g_prof.ev[2 * i + 1]) != cudaSuccess)
      return TP_ERR_CUDA;
    float ms = 0.0f;
    if (cudaEventElapsedTime(&ms, g_prof.ev[2 * i], g_prof.ev[2 * i + 1]) !=
        cudaSuccess)
      return TP_ERR_CUDA;
    r.launches += 1;
    r.ms += ms;
    r.flops += g_prof.rec[i].flops;
    r.bytes += g_prof.rec[i].bytes;
  }
  *out = r;
  return TP_OK;
}

// --------------------------------------------------------------- status --
extern "C" tp_status tp_device_status(tp_stream stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return TP_ERR_CUDA;
  unsigned* p = device_status_ptr();
  if (p == nullptr) return TP_ERR_CUDA;
  unsigned h[4] = {0, 0, 0, 0};
  if (cudaMemcpy(h, p, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess)
    return TP_ERR_CUDA;
  if (h[0] != 0) {
    const unsigned zero[4] = {0, 0, 0, 0};
    if (cudaMemcpy(p, zero, sizeof(zero), cudaMemcpyHostToDevice) !=
        cudaSuccess)
      return TP_ERR_CUDA;
    return h[0] == kDevRange ? TP_ERR_RANGE : TP_ERR_DEVICE_TIMEOUT;
  }
  return TP_OK;
}

extern "C" const char* tp_status_string(tp_status s) {
  switch (s) {
    case TP_OK: return "ok";
    case TP_ERR_NULL: return "required pointer is NULL";
    case TP_ERR_SHAPE: return "invalid or non-divisible shape";
    case TP_ERR_DTYPE: return "unknown dtype, activation, mode or scope";
    case TP_ERR_WORKSPACE: return "workspace or scratch too small";
    case TP_ERR_UNSUPPORTED: return "combination not supported";
    case TP_ERR_CUDA: return "CUDA call failed";
    case TP_ERR_DEVICE_TIMEOUT: return "a bounded device wait timed out";
    case TP_ERR_ARG: return "misaligned pointer or bad argument";
    case TP_ERR_RANGE: return "an attention-core operand exceeded the fp16 range";
  }
  return "unknown status";
}

extern "C" uint64_t tp_launch_count(void) { return g_launches.load(); }

extern "C" tp_status tp_selftest_wait_timeout(tp_stream stream) {
  return guarded([&]() -> tp_status {
    unsigned* st = device_status_ptr();
    if (st == nullptr) return TP_ERR_CUDA;
    return cuda_status(selftest_wait_timeout(st, stream));
  });
}

extern "C" int32_t tp_last_cuda_error(const char** name) {
  const int e = g_last_cuda_error.load();
  if (name != nullptr)
    *name = cudaGetErrorName(static_cast<cudaError_t>(e));
  return e;
}

extern "C" size_t tp_attn_set_ds_budget(size_t bytes) {
  return (size_t)attn_set_ds_budget(
      bytes > (size_t)INT64_MAX ? INT64_MAX : (int64_t)bytes);
}

extern "C" int32_t tp_num_sms(void) {
  int n = 0;
  if (cudaGetDeviceCount(&n) != cudaSuccess || n == 0) return 0;
  return device_sm_count();
}

// ----------------------------------------------------------------- layer --
// The pre-norm layer composed from the block entry points on one stream.
namespace {

tp_status check_layer(const tp_layer_desc* d) {
  if (d == nullptr) return TP_ERR_NULL;
  if (d->dtype != TP_BF16 && d->dtype != TP_FP8) return TP_ERR_UNSUPPORTED;
  if (!(d->eps > 0.0f)) return TP_ERR_ARG;
  if (d->h > 16384) return TP_ERR_SHAPE;   // the RMSNorm kernels' limit
  return TP_OK;
}

tp_attn_desc layer_attn(const tp_layer_desc* d) {
  tp_attn_desc a;
  a.b = d->b;
  a.s = d->s;
  a.h = d->h;
  a.n_q = d->n_q;
  a.n_kv = d->n_kv;
  a.d = d->d;
  a.n = d->n;
  a.dtype = d->dtype;
  a.causal = 1;
  a.mode = d->mode;
  return a;
}

tp_mlp_desc layer_mlp(const tp_layer_desc* d) {
  tp_mlp_desc m;
  m.T = d->b * d->s;
  m.h = d->h;
  m.h_ffn = d->h_ffn;
  m.n = d->n;
  m.dtype = d->dtype;
  m.act = TP_SWIGLU;
  m.mode = d->mode;
  m.dropout_p = 0.0f;
  m.seed = 0;
  return m;
}

struct LayerFwdLayout {
  void *xn1 = nullptr, *x1 = nullptr, *xn2 = nullptr;
  float *rstd1 = nullptr, *rstd2 = nullptr;
  void *attn_ws = nullptr, *mlp_ws = nullptr;
  // bf16 mode: fp16 copies of the first norm's output and of [Wq; Wk; Wv]
  // stacked, the operands of the Q, K, V projections (forward only)
  void *xn1h = nullptr, *wqkvh = nullptr;
  size_t attn_bytes = 0, mlp_bytes = 0, bytes = 0;
};

// Zero `bytes` when a block rejects its part of the desc.
LayerFwdLayout layer_fwd_layout(const tp_layer_desc* d, void* ws) {
  LayerFwdLayout L;
  const tp_attn_desc ad = layer_attn(d);
  const tp_mlp_desc md = layer_mlp(d);
  L.attn_bytes = tp_attn_workspace_bytes(&ad);
  L.mlp_bytes = tp_mlp_workspace_bytes(&md);
  if (L.attn_bytes == 0 || L.mlp_bytes == 0) return L;
  Carver c(ws);
  const size_t th = (size_t)(d->b * d->s) * (size_t)d->h * 2;
  L.xn1 = c.take(th);
  L.x1 = c.take(th);
  L.xn2 = c.take(th);
  L.rstd1 = static_cast<float*>(c.take((size_t)(d->b * d->s) * 4));
  L.rstd2 = static_cast<float*>(c.take((size_t)(d->b * d->s) * 4));
  L.attn_ws = c.take(L.attn_bytes);
  L.mlp_ws = c.take(L.mlp_bytes);
  if (d->dtype == TP_BF16) {
    const size_t qd = (size_t)d->n_q * d->d, kd = (size_t)d->n_kv * d->d;
    L.xn1h = c.take(th);
    L.wqkvh = c.take((qd + 2 * kd) * (size_t)d->h * 2);
  }
  L.bytes = c.off;
  return L;
}

struct LayerBwdLayout {
  void *dxn = nullptr, *dx1 = nullptr, *norm = nullptr, *blk = nullptr;
  size_t norm_bytes = 0, blk_bytes = 0, bytes = 0;
};

LayerBwdLayout layer_bwd_layout(const tp_layer_desc* d, void* scratch) {
  LayerBwdLayout L;
  const tp_attn_desc ad = layer_attn(d);
  const tp_mlp_desc md = layer_mlp(d);
  const size_t a = tp_attn_bwd_scratch_bytes(&ad);
  const size_t m = tp_mlp_bwd_scratch_bytes(&md);
  L.norm_bytes = tp_rmsnorm_bwd_scratch_bytes(d->b * d->s, d->h);
  if (a == 0 || m == 0 || L.norm_bytes == 0) return L;
  L.blk_bytes = std::max(a, m);
  Carver c(scratch);
  const size_t th = (size_t)(d->b * d->s) * (size_t)d->h * 2;
  L.dxn = c.take(th);
  L.dx1 = c.take(th);
  L.norm = c.take(L.norm_bytes);
  L.blk = c.take(L.blk_bytes);
  L.bytes = c.off;
  return L;
}

}  // namespace

extern "C" size_t tp_layer_workspace_bytes(const tp_layer_desc* d) {
  if (check_layer(d) != TP_OK) return 0;
  return layer_fwd_layout(d, nullptr).bytes;
}

extern "C" size_t tp_layer_bwd_scratch_bytes(const tp_layer_desc* d) {
  if (check_layer(d) != TP_OK) return 0;
  return layer_bwd_layout(d, nullptr).bytes;
}

extern "C" tp_status tp_layer_fwd(const tp_layer_desc* d, const void* x,
                                  const void* g1, const void* Wq,
                                  const void* Wk, const void* Wv,
                                  const void* Wo, const void* g2,
                                  const void* W1, const void* W2, void* out,
                                  void* ws, size_t ws_bytes,
                                  tp_stream stream) {
  return guarded([&]() -> tp_status {
    tp_status st = check_layer(d);
    if (st != TP_OK) return st;
    if (!x || !g1 || !g2 || !out || !ws) return TP_ERR_NULL;
    const LayerFwdLayout L = layer_fwd_layout(d, ws);
    if (L.bytes == 0) {   // a block rejects the shape: report its reason
      const tp_attn_desc ad = layer_attn(d);
      const tp_mlp_desc md = layer_mlp(d);
      st = check_attn(&ad);
      return st != TP_OK ? st : check_mlp(&md);
    }
    if (ws_bytes < L.bytes) return TP_ERR_WORKSPACE;
    if (!Wq || !Wk || !Wv || !Wo || !W1 || !W2) return TP_ERR_NULL;
    if (!aligned16(x) || !aligned16(g1) || !aligned16(g2) || !aligned16(Wq) ||
        !aligned16(Wk) || !aligned16(Wv) || !aligned16(Wo) ||
        !aligned16(W1) || !aligned16(W2) || !aligned16(out) || !aligned16(ws))
      return TP_ERR_ARG;
    const int64_t T = d->b * d->s, h = d->h;
    const tp_attn_desc ad = layer_attn(d);
    const tp_mlp_desc md = layer_mlp(d);
    if (d->dtype == TP_BF16) {
      // the first norm writes its output in bf16 (saved for the backward)
      // and fp16 (the Q, K, V projections' operand, with fp16 weights)
      unsigned* status = device_status_ptr();
      const int64_t qd = (int64_t)d->n_q * d->d, kd = (int64_t)d->n_kv * d->d;
      int err = rmsnorm_fwd<__nv_bfloat16>(x, g1, L.xn1, L.rstd1, T, h, d->eps,
                                           stream, L.xn1h, status);
      // [Wq; Wk; Wv] stacked in fp16, one launch
      const void* wsrc[3] = {Wq, Wk, Wv};
      const int64_t wn[3] = {qd * h, kd * h, kd * h};
      if (!err) err = convert_f16(wsrc, wn, 3, L.wqkvh, status, stream);
      if (err) return cuda_status(err);
      QkvF16 f16in;
      f16in.x = L.xn1h;
      f16in.wqkv = L.wqkvh;
      const bool sp = d->mode == TP_REDUCE_SP;
      void* partials = nullptr;
      st = attn_fwd_impl(&ad, L.xn1, Wq, Wk, Wv, Wo, nullptr, x, L.x1,
                         L.attn_ws, L.attn_bytes, stream, &f16in,
                         sp ? &partials : nullptr);
      if (st == TP_OK && sp) {
        // reduce-scatter of the attention partials + residual, then the
        // second RMSNorm on the same rows; the all-gathered xn2 is the
        // MLP's input
        int err = reduce_norm_fwd<__nv_bfloat16>(
            partials, d->n, T * h, nullptr, x, L.x1, DropoutSpec(), g2,
            L.xn2, nullptr, L.rstd2, T, h, d->eps, status, stream);
        if (err) return cuda_status(err);
        return tp_mlp_fwd(&md, L.xn2, W1, nullptr, W2, nullptr, L.x1, out,
                          L.mlp_ws, L.mlp_bytes, stream);
      }
    } else {
      st = tp_rmsnorm_fwd(T, h, d->eps, TP_BF16, x, g1, L.xn1, L.rstd1,
                          stream);
      if (st == TP_OK)
        st = tp_attn_fwd(&ad, L.xn1, Wq, Wk, Wv, Wo, nullptr, x, L.x1,
                         L.attn_ws, L.attn_bytes, stream);
    }
    if (st == TP_OK)
      st = tp_rmsnorm_fwd(T, h, d->eps, TP_BF16, L.x1, g2, L.xn2, L.rstd2,
                          stream);
    if (st == TP_OK)
      st = tp_mlp_fwd(&md, L.xn2, W1, nullptr, W2, nullptr, L.x1, out,
                      L.mlp_ws, L.mlp_bytes, stream);
    return st;
  });
}

extern "C" tp_status tp_layer_bwd(const tp_layer_desc* d, const void* dout,
                                  const void* x, const void* g1,
                                  const void* Wq, const void* Wk,
                                  const void* Wv, const void* Wo,
                                  const void* g2, const void* W1,
                                  const void* W2, const void* ws, void* dx,
                                  void* dg1, void* dWq, void* dWk, void* dWv,
                                  void* dWo, void* dg2, void* dW1, void* dW2,
                                  void* scratch, size_t scratch_bytes,
                                  tp_stream stream) {
  return guarded([&]() -> tp_status {
    tp_status st = check_layer(d);
    if (st != TP_OK) return st;
    if (!dout || !x || !g1 || !g2 || !ws || !dx || !dg1 || !dg2 || !scratch)
      return TP_ERR_NULL;
    const LayerFwdLayout F = layer_fwd_layout(d, const_cast<void*>(ws));
    const LayerBwdLayout L = layer_bwd_layout(d, scratch);
    if (F.bytes == 0 || L.bytes == 0) return TP_ERR_SHAPE;
    if (scratch_bytes < L.bytes) return TP_ERR_WORKSPACE;
    const int64_t T = d->b * d->s, h = d->h;
    const tp_attn_desc ad = layer_attn(d);
    const tp_mlp_desc md = layer_mlp(d);
    if (d->mode == TP_REDUCE_SP) {
      // each f reduction (the blocks' input-gradient partials) is summed
      // inside the RMSNorm backward of the rows it feeds
      if (!Wq || !Wk || !Wv || !Wo || !W1 || !W2 || !dWq || !dWk || !dWv ||
          !dWo || !dW1 || !dW2)
        return TP_ERR_NULL;
      void* partials = nullptr;
      st = mlp_bwd_impl(&md, dout, F.xn2, W1, W2, F.mlp_ws, nullptr, L.dxn,
                        dW1, nullptr, dW2, nullptr, L.blk, L.blk_bytes,
                        stream, &partials);
      if (st != TP_OK) return st;
      int err = rmsnorm_bwd_sum<__nv_bfloat16>(
          partials, d->n, T * h, F.x1, g2, F.rstd2, dout, L.dx1, dg2,
          static_cast<float*>(L.norm), T, h, stream, device_status_ptr());
      if (err) return cuda_status(err);
      st = attn_bwd_impl(&ad, L.dx1, F.xn1, Wq, Wk, Wv, Wo, F.attn_ws,
                         nullptr, L.dxn, dWq, dWk, dWv, dWo, nullptr, L.blk,
                         L.blk_bytes, stream, &partials);
      if (st != TP_OK) return st;
      err = rmsnorm_bwd_sum<__nv_bfloat16>(
          partials, d->n, T * h, x, g1, F.rstd1, L.dx1, dx, dg1,
          static_cast<float*>(L.norm), T, h, stream, device_status_ptr());
      return cuda_status(err);
    }
    // MLP block: d(xn2) into dxn, then RMSNorm₂ with the residual's dout
    st = tp_mlp_bwd(&md, dout, F.xn2, W1, W2, F.mlp_ws, nullptr, L.dxn, dW1,
                    nullptr, dW2, nullptr, L.blk, L.blk_bytes, stream);
    if (st == TP_OK)
      st = tp_rmsnorm_bwd(T, h, d->eps, TP_BF16, L.dxn, F.x1, g2, F.rstd2,
                          dout, L.dx1, dg2, L.norm, L.norm_bytes, stream);
    // attention block: d(xn1) into dxn, then RMSNorm₁ with dx1 as residual
    if (st == TP_OK)
      st = tp_attn_bwd(&ad, L.dx1, F.xn1, Wq, Wk, Wv, Wo, F.attn_ws, nullptr,
                       L.dxn, dWq, dWk, dWv, dWo, nullptr, L.blk, L.blk_bytes,
                       stream);
    if (st == TP_OK)
      st = tp_rmsnorm_bwd(T, h, d->eps, TP_BF16, L.dxn, x, g1, F.rstd1, L.dx1,
                          dx, dg1, L.norm, L.norm_bytes, stream);
    return st;
  });
}
