"""Thin ctypes binding of ``libtp.so`` (declared in include/tp.h).

Argument marshalling only: torch tensors are passed as raw device pointers,
the caller's current CUDA stream as the stream handle, and every status code
is turned into a ``TPError``.  All computation happens in the library's CUDA
kernels; there is no fallback — if the library has not been built, ``lib()``
raises.
"""

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libtp.so")

F32, BF16, FP8 = 0, 1, 2
GELU, SWIGLU = 0, 1
FUSED, MATERIALISED, OVERLAP, SP = 0, 1, 2, 3
SCOPE_MLP, SCOPE_ATTN, SCOPE_LAYER = 0, 1, 2

STATUS = {0: "TP_OK", 1: "TP_ERR_NULL", 2: "TP_ERR_SHAPE", 3: "TP_ERR_DTYPE",
          4: "TP_ERR_WORKSPACE", 5: "TP_ERR_UNSUPPORTED", 6: "TP_ERR_CUDA",
          7: "TP_ERR_DEVICE_TIMEOUT", 8: "TP_ERR_ARG", 9: "TP_ERR_RANGE"}


class TPError(RuntimeError):
    def __init__(self, code, where, detail=""):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)}{detail}")


class MlpDesc(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("h", ctypes.c_int64),
                ("h_ffn", ctypes.c_int64), ("n", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("act", ctypes.c_int32),
                ("mode", ctypes.c_int32), ("dropout_p", ctypes.c_float),
                ("seed", ctypes.c_uint64)]


class AttnDesc(ctypes.Structure):
    _fields_ = [("b", ctypes.c_int64), ("s", ctypes.c_int64),
                ("h", ctypes.c_int64), ("n_q", ctypes.c_int32),
                ("n_kv", ctypes.c_int32), ("d", ctypes.c_int32),
                ("n", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("causal", ctypes.c_int32), ("mode", ctypes.c_int32)]


class CommReport(ctypes.Structure):
    _fields_ = [(k, ctypes.c_uint64) for k in (
        "reductions_fwd", "reductions_bwd", "payload_bytes", "ring_bytes_num",
        "ring_bytes_den", "page2_bytes", "total_payload", "total_ring_num",
        "total_page2", "sp_rs_bytes_num", "sp_ag_bytes_num", "sp_bytes_den",
        "sp_reduce_scatters", "sp_all_gathers", "sp_total_num")]


class ActDesc(ctypes.Structure):
    _fields_ = [("b", ctypes.c_int64), ("s", ctypes.c_int64),
                ("h", ctypes.c_int64), ("h_ffn", ctypes.c_int64),
                ("n_q", ctypes.c_int32), ("n_kv", ctypes.c_int32),
                ("d", ctypes.c_int32), ("n", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("act", ctypes.c_int32),
                ("dropout", ctypes.c_int32), ("seq_parallel", ctypes.c_int32)]


class ActReport(ctypes.Structure):
    _fields_ = [(k, ctypes.c_uint64) for k in (
        "mlp_x", "mlp_hidden", "mlp_act", "mlp_mask", "attn_x", "attn_q",
        "attn_kv", "attn_scores", "attn_lse", "attn_o", "norm_x", "norm_rstd",
        "mlp_bytes", "attn_bytes_pages", "attn_bytes_flash",
        "layer_bytes_flash")]


class LayerDesc(ctypes.Structure):
    _fields_ = [("b", ctypes.c_int64), ("s", ctypes.c_int64),
                ("h", ctypes.c_int64), ("h_ffn", ctypes.c_int64),
                ("n_q", ctypes.c_int32), ("n_kv", ctypes.c_int32),
                ("d", ctypes.c_int32), ("n", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("mode", ctypes.c_int32),
                ("eps", ctypes.c_float)]


class ProfileEntry(ctypes.Structure):
    _fields_ = [("launches", ctypes.c_uint64), ("ms", ctypes.c_double),
                ("flops", ctypes.c_double), ("bytes", ctypes.c_double)]


KERNEL_FAMILIES = ["gemm_tc", "gemm_simt", "attn_fwd", "attn_bwd_dkdv",
                   "attn_bwd_dq", "reduce", "elementwise", "rmsnorm",
                   "gemm_tc_fp8", "quantize_fp8"]

_P = ctypes.c_void_p
_I64, _I32, _F, _SZ, _U64 = (ctypes.c_int64, ctypes.c_int32, ctypes.c_float,
                             ctypes.c_size_t, ctypes.c_uint64)
_MP = ctypes.POINTER(MlpDesc)
_AP = ctypes.POINTER(AttnDesc)
_LP = ctypes.POINTER(LayerDesc)
_U64P = ctypes.POINTER(ctypes.c_uint64)

# name -> (restype, argtypes); mirrors include/tp.h
SIGNATURES = {
    "tp_mlp_workspace_bytes": (_SZ, [_MP]),
    "tp_mlp_bwd_scratch_bytes": (_SZ, [_MP]),
    "tp_mlp_fwd": (_I32, [_MP, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "tp_mlp_bwd": (_I32, [_MP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                          _P, _SZ, _P]),
    "tp_attn_workspace_bytes": (_SZ, [_AP]),
    "tp_attn_bwd_scratch_bytes": (_SZ, [_AP]),
    "tp_attn_set_ds_budget": (_SZ, [_SZ]),
    "tp_attn_fwd": (_I32, [_AP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "tp_attn_bwd": (_I32, [_AP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P,
                           _P, _P, _P, _P, _SZ, _P]),
    "tp_layer_workspace_bytes": (_SZ, [_LP]),
    "tp_layer_bwd_scratch_bytes": (_SZ, [_LP]),
    "tp_layer_fwd": (_I32, [_LP] + [_P] * 11 + [_SZ, _P]),
    "tp_layer_bwd": (_I32, [_LP] + [_P] * 21 + [_SZ, _P]),
    "tp_rmsnorm_fwd": (_I32, [_I64, _I64, _F, _I32, _P, _P, _P, _P, _P]),
    "tp_rmsnorm_bwd_scratch_bytes": (_SZ, [_I64, _I64]),
    "tp_rmsnorm_bwd": (_I32, [_I64, _I64, _F, _I32, _P, _P, _P, _P, _P, _P,
                              _P, _P, _SZ, _P]),
    "tp_rmsnorm_bwd_noalloc": (_I32, [_I64, _I64, _F, _I32, _P, _P, _P, _P,
                                      _P, _P, _P, _P]),
    "tp_comm_bytes": (_I32, [_I32, _I64, _I64, _I32, _I32,
                             ctypes.POINTER(CommReport)]),
    "tp_act_memory": (_I32, [ctypes.POINTER(ActDesc),
                             ctypes.POINTER(ActReport)]),
    "tp_quantize_fp8": (_I32, [_I64, _P, _P, _P, _P, _P]),
    "tp_gemm_fp8": (_I32, [_I64, _I64, _I64, _P, _I64, _P, _P, _I64, _P, _P,
                           _I64, _P]),
    "tp_mlp_flops": (_I32, [_MP, _U64P, _U64P]),
    "tp_attn_flops": (_I32, [_AP, _U64P, _U64P]),
    "tp_gemm": (_I32, [_I32, _I64, _I64, _I64, _P, _I64, _I32, _P, _I64, _I32,
                       _P, _I64, _P]),
    "tp_profile_enable": (_I32, [_I32]),
    "tp_profile_reset": (_I32, []),
    "tp_profile_read": (_I32, [_I32, ctypes.POINTER(ProfileEntry)]),
    "tp_device_status": (_I32, [_P]),
    "tp_status_string": (ctypes.c_char_p, [_I32]),
    "tp_launch_count": (_U64, []),
    "tp_last_cuda_error": (_I32, [ctypes.POINTER(ctypes.c_char_p)]),
    "tp_selftest_wait_timeout": (_I32, [_P]),
    "tp_num_sms": (_I32, []),
}

_lib = None


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "megatron_tensor_transformer_gate_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def check(code, where):
    if code != 0:
        detail = ""
        if code == 6:   # TP_ERR_CUDA: name the CUDA error behind it
            name = ctypes.c_char_p()
            err = lib().tp_last_cuda_error(ctypes.byref(name))
            detail = f" ({err}: {(name.value or b'').decode()})"
        raise TPError(code, where, detail)


def ptr(t):
    """Device (or host) address of a tensor, or None."""
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def stream_handle(stream=None):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def dtype_code(t):
    import torch
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


# ------------------------------------------------------------ accounting --
def comm_bytes(scope, T, h, n, dtype):
    r = CommReport()
    check(lib().tp_comm_bytes(scope, T, h, n, dtype, ctypes.byref(r)),
          "tp_comm_bytes")
    return {k: getattr(r, k) for k, _ in CommReport._fields_}


def quantize_fp8(x, q, scale, amax_work, stream=None):
    """E4M3 codes of the bf16 tensor x into q (uint8, same numel); the
    per-tensor scale into the one-element fp32 tensor ``scale``."""
    check(lib().tp_quantize_fp8(x.numel(), ptr(x), ptr(q), ptr(scale),
                                ptr(amax_work), stream_handle(stream)),
          "tp_quantize_fp8")


def selftest_wait_timeout(stream=None):
    """Enqueue the kernel whose bounded wait runs out (about 2 s)."""
    check(lib().tp_selftest_wait_timeout(stream_handle(stream)),
          "tp_selftest_wait_timeout")


def gemm_fp8(qa, scale_a, qb, scale_b, C, stream=None):
    """C[M, N] = qa·qbᵀ / (scale_a·scale_b) on E4M3 codes (K-major both)."""
    M, N = C.shape
    K = qa.shape[1]
    check(lib().tp_gemm_fp8(M, N, K, ptr(qa), qa.stride(0), ptr(scale_a),
                            ptr(qb), qb.stride(0), ptr(scale_b), ptr(C),
                            C.stride(0), stream_handle(stream)),
          "tp_gemm_fp8")


def act_memory(b, s, h, h_ffn, n_q, n_kv, d, n, dtype=BF16, act=SWIGLU,
               dropout=False, seq_parallel=False):
    """Saved activations per rank (elements by tensor, bytes by block)."""
    r = ActReport()
    desc = ActDesc(b, s, h, h_ffn, n_q, n_kv, d, n, dtype, act, int(dropout),
                   int(seq_parallel))
    check(lib().tp_act_memory(ctypes.byref(desc), ctypes.byref(r)),
          "tp_act_memory")
    return {k: getattr(r, k) for k, _ in ActReport._fields_}


def mlp_flops(desc):
    f, b = ctypes.c_uint64(), ctypes.c_uint64()
    check(lib().tp_mlp_flops(ctypes.byref(desc), ctypes.byref(f),
                             ctypes.byref(b)), "tp_mlp_flops")
    return f.value, b.value


def attn_flops(desc):
    f, b = ctypes.c_uint64(), ctypes.c_uint64()
    check(lib().tp_attn_flops(ctypes.byref(desc), ctypes.byref(f),
                              ctypes.byref(b)), "tp_attn_flops")
    return f.value, b.value


# ------------------------------------------------------------------ GEMM --
def gemm(A, B, C, a_mn_major=False, b_mn_major=False, stream=None):
    """C[M, N] = A·Bᵀ with the operand layouts of tp_gemm."""
    M, N = C.shape
    K = A.shape[0] if a_mn_major else A.shape[1]
    check(lib().tp_gemm(dtype_code(C), M, N, K, ptr(A), A.stride(0),
                        int(a_mn_major), ptr(B), B.stride(0), int(b_mn_major),
                        ptr(C), C.stride(0), stream_handle(stream)),
          "tp_gemm")


# ------------------------------------------------------------------- MLP --
def mlp_desc(T, h, h_ffn, n, dtype=BF16, act=GELU, mode=FUSED, dropout_p=0.0,
             seed=0):
    return MlpDesc(T, h, h_ffn, n, dtype, act, mode, dropout_p, seed)


def mlp_workspace_bytes(desc):
    return lib().tp_mlp_workspace_bytes(ctypes.byref(desc))


def mlp_bwd_scratch_bytes(desc):
    return lib().tp_mlp_bwd_scratch_bytes(ctypes.byref(desc))


def mlp_fwd(desc, X, W1, W2, Out, ws, b1=None, b2=None, R=None, stream=None):
    check(lib().tp_mlp_fwd(ctypes.byref(desc), ptr(X), ptr(W1), ptr(b1),
                           ptr(W2), ptr(b2), ptr(R), ptr(Out), ptr(ws),
                           ws.numel() * ws.element_size(),
                           stream_handle(stream)), "tp_mlp_fwd")


def mlp_bwd(desc, dOut, X, W1, W2, ws, dX, dW1, dW2, scratch, db1=None,
            db2=None, dres=None, stream=None):
    check(lib().tp_mlp_bwd(ctypes.byref(desc), ptr(dOut), ptr(X), ptr(W1),
                           ptr(W2), ptr(ws), ptr(dres), ptr(dX), ptr(dW1),
                           ptr(db1), ptr(dW2), ptr(db2), ptr(scratch),
                           scratch.numel() * scratch.element_size(),
                           stream_handle(stream)), "tp_mlp_bwd")


# ------------------------------------------------------------- attention --
def attn_desc(b, s, h, n_q, n_kv, d, n, dtype=BF16, causal=True, mode=FUSED):
    return AttnDesc(b, s, h, n_q, n_kv, d, n, dtype, int(causal), mode)


def attn_workspace_bytes(desc):
    return lib().tp_attn_workspace_bytes(ctypes.byref(desc))


def attn_bwd_scratch_bytes(desc):
    return lib().tp_attn_bwd_scratch_bytes(ctypes.byref(desc))


def attn_set_ds_budget(nbytes):
    """Bound on the attention backward's dS tile bytes per pass (0 = the
    default); returns the previous bound."""
    return lib().tp_attn_set_ds_budget(nbytes)


def attn_fwd(desc, X, Wq, Wk, Wv, Wo, Out, ws, bo=None, R=None, stream=None):
    check(lib().tp_attn_fwd(ctypes.byref(desc), ptr(X), ptr(Wq), ptr(Wk),
                            ptr(Wv), ptr(Wo), ptr(bo), ptr(R), ptr(Out),
                            ptr(ws), ws.numel() * ws.element_size(),
                            stream_handle(stream)), "tp_attn_fwd")


def attn_bwd(desc, dOut, X, Wq, Wk, Wv, Wo, ws, dX, dWq, dWk, dWv, dWo,
             scratch, dbo=None, dres=None, stream=None):
    check(lib().tp_attn_bwd(ctypes.byref(desc), ptr(dOut), ptr(X), ptr(Wq),
                            ptr(Wk), ptr(Wv), ptr(Wo), ptr(ws), ptr(dres),
                            ptr(dX), ptr(dWq), ptr(dWk), ptr(dWv), ptr(dWo),
                            ptr(dbo), ptr(scratch),
                            scratch.numel() * scratch.element_size(),
                            stream_handle(stream)), "tp_attn_bwd")


# --------------------------------------------------------------- RMSNorm --
# ----------------------------------------------------------------- layer --
def layer_desc(b, s, h, h_ffn, n_q, n_kv, d, n, dtype=BF16, mode=FUSED,
               eps=1e-5):
    return LayerDesc(b, s, h, h_ffn, n_q, n_kv, d, n, dtype, mode, eps)


def layer_workspace_bytes(desc):
    return lib().tp_layer_workspace_bytes(ctypes.byref(desc))


def layer_bwd_scratch_bytes(desc):
    return lib().tp_layer_bwd_scratch_bytes(ctypes.byref(desc))


def layer_fwd(desc, x, P, out, ws, stream=None):
    """out = x1 + MLP(RMSNorm₂(x1)), x1 = x + Attn(RMSNorm₁(x)); P holds g1,
    Wq, Wk, Wv, Wo, g2, W1, W2."""
    check(lib().tp_layer_fwd(
        ctypes.byref(desc), ptr(x), *(ptr(P[k]) for k in
                                      ("g1", "Wq", "Wk", "Wv", "Wo", "g2",
                                       "W1", "W2")),
        ptr(out), ptr(ws), ws.numel() * ws.element_size(),
        stream_handle(stream)), "tp_layer_fwd")


def layer_bwd(desc, dout, x, P, ws, grads, scratch, stream=None):
    """grads: dX, dg1, dWq, dWk, dWv, dWo, dg2, dW1, dW2 (overwritten)."""
    names = ("g1", "Wq", "Wk", "Wv", "Wo", "g2", "W1", "W2")
    check(lib().tp_layer_bwd(
        ctypes.byref(desc), ptr(dout), ptr(x), *(ptr(P[k]) for k in names),
        ptr(ws), ptr(grads["dX"]), *(ptr(grads["d" + k]) for k in names),
        ptr(scratch), scratch.numel() * scratch.element_size(),
        stream_handle(stream)), "tp_layer_bwd")


def rmsnorm_fwd(x, gamma, y, rstd, eps=1e-5, stream=None):
    T, h = x.shape
    check(lib().tp_rmsnorm_fwd(T, h, eps, dtype_code(x), ptr(x), ptr(gamma),
                               ptr(y), ptr(rstd), stream_handle(stream)),
          "tp_rmsnorm_fwd")


def rmsnorm_bwd_scratch_bytes(T, h):
    return lib().tp_rmsnorm_bwd_scratch_bytes(T, h)


def rmsnorm_bwd(dy, x, gamma, rstd, dx, dgamma, scratch, dres=None, eps=1e-5,
                stream=None):
    T, h = x.shape
    check(lib().tp_rmsnorm_bwd(T, h, eps, dtype_code(x), ptr(dy), ptr(x),
                               ptr(gamma), ptr(rstd), ptr(dres), ptr(dx),
                               ptr(dgamma), ptr(scratch),
                               scratch.numel() * scratch.element_size(),
                               stream_handle(stream)), "tp_rmsnorm_bwd")


def rmsnorm_bwd_noalloc(dy, x, gamma, rstd, dx, dgamma, dres=None, eps=1e-5,
                        stream=None):
    """RMSNorm backward without caller scratch (see tp_rmsnorm_bwd_noalloc)."""
    T, h = x.shape
    check(lib().tp_rmsnorm_bwd_noalloc(T, h, eps, dtype_code(x), ptr(dy),
                                       ptr(x), ptr(gamma), ptr(rstd),
                                       ptr(dres), ptr(dx), ptr(dgamma),
                                       stream_handle(stream)),
          "tp_rmsnorm_bwd_noalloc")


def device_status(stream=None):
    check(lib().tp_device_status(stream_handle(stream)), "tp_device_status")


def launch_count():
    return lib().tp_launch_count()


# ------------------------------------------------------------- profiling --
def profile_enable(max_launches):
    check(lib().tp_profile_enable(max_launches), "tp_profile_enable")


def profile_reset():
    check(lib().tp_profile_reset(), "tp_profile_reset")


def profile_read():
    """{family: {launches, ms, flops, bytes}} for every kernel family."""
    out = {}
    for i, name in enumerate(KERNEL_FAMILIES):
        e = ProfileEntry()
        check(lib().tp_profile_read(i, ctypes.byref(e)), "tp_profile_read")
        out[name] = {"launches": e.launches, "ms": e.ms, "flops": e.flops,
                     "bytes": e.bytes}
    return out
