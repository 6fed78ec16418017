"""Convenience wrappers that own the workspaces of the TP block calls.

PyTorch only provides device memory here; every step runs in ``libtp.so``.
``TPMLP`` / ``TPAttention`` hold the forward workspace (saved activations)
and the backward scratch for one shape; ``TPLayer`` composes the pre-norm
layer  x1 = x + Attn(RMSNorm₁(x)),  out = x1 + MLP(RMSNorm₂(x1))  out of the
library's RMSNorm, attention and MLP entry points, which gives the layer's
four TP reductions (attention g and MLP g in forward, MLP f and attention f
in backward).
"""

import torch

from . import binding as B

_TD = {B.F32: torch.float32, B.BF16: torch.bfloat16,
       B.FP8: torch.bfloat16}   # FP8 mode stores bf16 tensors


def _buf(nbytes, device):
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)


def _views(ws, specs):
    """Tensors viewing consecutive 256-byte-aligned regions of a workspace
    (the layout include/tp.h documents); specs = [(name, shape, dtype)]."""
    out, off = {}, 0
    for name, shape, dt in specs:
        off = (off + 255) // 256 * 256
        n = 1
        for d in shape:
            n *= d
        nbytes = n * torch.empty((), dtype=dt).element_size()
        out[name] = ws[off:off + nbytes].view(dt).view(*shape)
        off += nbytes
    return out


class TPMLP:
    def __init__(self, T, h, h_ffn, n, *, dtype=B.BF16, act=B.GELU,
                 mode=B.FUSED, dropout_p=0.0, seed=0, device="cuda"):
        self.desc = B.mlp_desc(T, h, h_ffn, n, dtype, act, mode, dropout_p,
                               seed)
        self.T, self.h, self.f, self.act = T, h, h_ffn, act
        self.dtype = _TD[dtype]
        self.device = device
        self.ws = _buf(B.mlp_workspace_bytes(self.desc), device)
        self.scratch = _buf(B.mlp_bwd_scratch_bytes(self.desc), device)

    def forward(self, X, W1, W2, b1=None, b2=None, R=None, out=None,
                stream=None):
        if out is None:
            out = torch.empty((self.T, self.h), dtype=self.dtype,
                              device=self.device)
        B.mlp_fwd(self.desc, X, W1, W2, out, self.ws, b1=b1, b2=b2, R=R,
                  stream=stream)
        return out

    def backward(self, dOut, X, W1, W2, dres=None, want_db1=False,
                 want_db2=False, grads=None, stream=None):
        g = grads if grads is not None else self.alloc_grads(W1, W2,
                                                             want_db1,
                                                             want_db2)
        B.mlp_bwd(self.desc, dOut, X, W1, W2, self.ws, g["dX"], g["dW1"],
                  g["dW2"], self.scratch, db1=g.get("db1"), db2=g.get("db2"),
                  dres=dres, stream=stream)
        return g

    def saved(self):
        """Views of the activations the forward call saved for backward."""
        tf = (self.T, self.f)
        names = ("H", "A") if self.act == B.GELU else ("G", "U", "A")
        return _views(self.ws, [(n, tf, self.dtype) for n in names])

    def alloc_grads(self, W1, W2, want_db1=False, want_db2=False):
        kw = dict(dtype=self.dtype, device=self.device)
        g = {"dX": torch.empty((self.T, self.h), **kw),
             "dW1": torch.empty_like(W1), "dW2": torch.empty_like(W2)}
        if want_db1:
            g["db1"] = torch.empty((W1.shape[0],), **kw)
        if want_db2:
            g["db2"] = torch.empty((self.h,), **kw)
        return g


class TPAttention:
    """dtype B.BF16, or B.FP8: the projections of the forward on E4M3
    operands (bf16 storage and backward)."""

    def __init__(self, b, s, h, n_q, n_kv, d, n, *, causal=True, mode=B.FUSED,
                 dtype=B.BF16, device="cuda"):
        self.desc = B.attn_desc(b, s, h, n_q, n_kv, d, n, dtype, causal,
                                mode)
        self.T, self.h = b * s, h
        self.shape = (b, s, n_q, n_kv, d)
        self.device = device
        self.ws = _buf(B.attn_workspace_bytes(self.desc), device)
        self.scratch = _buf(B.attn_bwd_scratch_bytes(self.desc), device)

    def forward(self, X, Wq, Wk, Wv, Wo, bo=None, R=None, out=None,
                stream=None):
        if out is None:
            out = torch.empty((self.T, self.h), dtype=torch.bfloat16,
                              device=self.device)
        B.attn_fwd(self.desc, X, Wq, Wk, Wv, Wo, out, self.ws, bo=bo, R=R,
                   stream=stream)
        return out

    def backward(self, dOut, X, Wq, Wk, Wv, Wo, dres=None, want_dbo=False,
                 grads=None, stream=None):
        g = grads if grads is not None else self.alloc_grads(Wq, Wk, Wv, Wo,
                                                             want_dbo)
        B.attn_bwd(self.desc, dOut, X, Wq, Wk, Wv, Wo, self.ws, g["dX"],
                   g["dWq"], g["dWk"], g["dWv"], g["dWo"], self.scratch,
                   dbo=g.get("dbo"), dres=dres, stream=stream)
        return g

    def saved(self):
        """Views of Q, K, V (fp16), O (bf16) and LSE saved by the forward."""
        b, s, nq, nkv, d = self.shape
        T = b * s
        return _views(self.ws, [("Q", (T, nq * d), torch.float16),
                                ("K", (T, nkv * d), torch.float16),
                                ("V", (T, nkv * d), torch.float16),
                                ("O", (T, nq * d), torch.bfloat16),
                                ("LSE", (b, nq, s), torch.float32)])

    def alloc_grads(self, Wq, Wk, Wv, Wo, want_dbo=False):
        g = {"dX": torch.empty((self.T, self.h), dtype=torch.bfloat16,
                               device=self.device),
             "dWq": torch.empty_like(Wq), "dWk": torch.empty_like(Wk),
             "dWv": torch.empty_like(Wv), "dWo": torch.empty_like(Wo)}
        if want_dbo:
            g["dbo"] = torch.empty((self.h,), dtype=torch.bfloat16,
                                   device=self.device)
        return g


class TPLayer:
    """Pre-norm layer: RMSNorm → attention (+x) → RMSNorm → SwiGLU MLP (+x1),
    one tp_layer_fwd / tp_layer_bwd call per direction.  dtype B.FP8 runs
    every projection of the forward on E4M3 operands."""

    def __init__(self, b, s, h, h_ffn, n_q, n_kv, d, n, *, eps=1e-5,
                 act=B.SWIGLU, mode=B.FUSED, dtype=B.BF16, device="cuda"):
        if act != B.SWIGLU:
            raise ValueError("the layer's MLP is SwiGLU")
        self.T, self.h, self.eps = b * s, h, eps
        self.device = device
        self.desc = B.layer_desc(b, s, h, h_ffn, n_q, n_kv, d, n, dtype, mode,
                                 eps)
        self.ws = _buf(B.layer_workspace_bytes(self.desc), device)
        self.scratch = _buf(B.layer_bwd_scratch_bytes(self.desc), device)

    def forward(self, x, P, out=None, stream=None):
        if out is None:
            out = torch.empty((self.T, self.h), dtype=torch.bfloat16,
                              device=self.device)
        B.layer_fwd(self.desc, x, P, out, self.ws, stream)
        return out

    def alloc_grads(self, P):
        g = {k: torch.empty_like(P[k]) for k in ("g1", "Wq", "Wk", "Wv", "Wo",
                                                 "g2", "W1", "W2")}
        g = {"d" + k: v for k, v in g.items()}
        g["dX"] = torch.empty((self.T, self.h), dtype=torch.bfloat16,
                              device=self.device)
        return g

    def backward(self, dout, x, P, grads=None, stream=None):
        g = grads if grads is not None else self.alloc_grads(P)
        B.layer_bwd(self.desc, dout, x, P, self.ws, g, self.scratch, stream)
        return g
