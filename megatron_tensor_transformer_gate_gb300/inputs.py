"""Seeded synthetic inputs for the tensor-parallel block workloads.

This module holds no arithmetic of the method: it only draws normal samples
with torch's counter-based generator and rounds them to the workload's dtype.
Both the CUDA path and the fp64 oracle receive the same rounded values (the
oracle converts them exactly to float64).

Workloads (shapes from the pages' notation: T = b·s tokens, hidden h,
intermediate h_ffn, heads n_q / n_kv of width d, TP degree n):

* ``mlp_gelu_f32``    GeLU MLP, fp32, b=1 s=64 h=128 h_ffn=512 n=2, no bias,
                      X, dOut ~ N(0,1), W ~ N(0, 1/fan_in) (variance).
* ``mlp_gelu_bf16``   GeLU MLP, bf16, b=4 s=1024 h=1024 h_ffn=4096 n=4, b2 ~
                      N(0, 0.02²), residual R = X, dropout p=0.1,
                      W ~ N(0, 0.02²).
* ``mlp_swiglu_bf16`` SwiGLU MLP, bf16, b=2 s=4096 h=4096 h_ffn=11008 n=8, no
                      bias, W ~ N(0, 1/fan_in) (std 1/√fan_in).
* ``attn_gqa_bf16``   causal GQA attention, bf16, b=2 s=2048 h=4096 n_q=32
                      n_kv=8 d=128 n=4, W ~ N(0, 0.02²).
* ``layer_bf16``      pre-norm layer (RMSNorm, GQA attention n_q=64 n_kv=8
                      d=128, SwiGLU h_ffn=28672), bf16, b=1 s=8192 h=8192
                      n=8, W ~ N(0, 0.02²), γ ~ 1 + N(0, 0.02²).

fan_in is the unsharded input width of the weight: h for W1/Wq/Wk/Wv, h_ffn
for W2, n_q·d for Wo.  Every tensor has its own sub-seed (base seed + a fixed
index), so a tensor's values do not depend on which others are drawn.
"""

import copy

import torch

WORKLOADS = {
    "mlp_gelu_f32": dict(kind="mlp", dtype="f32", b=1, s=64, h=128, h_ffn=512,
                         n=2, act="gelu", w_std="fan_in", b1=False, b2=False,
                         residual=None, p=0.0),
    "mlp_gelu_bf16": dict(kind="mlp", dtype="bf16", b=4, s=1024, h=1024,
                          h_ffn=4096, n=4, act="gelu", w_std=0.02, b1=False,
                          b2=True, residual="X", p=0.1),
    "mlp_swiglu_bf16": dict(kind="mlp", dtype="bf16", b=2, s=4096, h=4096,
                            h_ffn=11008, n=8, act="swiglu", w_std="fan_in",
                            b1=False, b2=False, residual=None, p=0.0),
    # the SwiGLU workload with its forward GEMMs on per-tensor scaled E4M3
    # (bf16 storage, bf16 backward)
    "mlp_swiglu_fp8": dict(kind="mlp", dtype="bf16", gemm_dtype="fp8", b=2,
                           s=4096, h=4096, h_ffn=11008, n=8, act="swiglu",
                           w_std="fan_in", b1=False, b2=False, residual=None,
                           p=0.0),
    "attn_gqa_bf16": dict(kind="attn", dtype="bf16", b=2, s=2048, h=4096,
                          n_q=32, n_kv=8, d=128, n=4, causal=True,
                          w_std=0.02, bo=False, residual=None),
    "layer_bf16": dict(kind="layer", dtype="bf16", b=1, s=8192, h=8192,
                       h_ffn=28672, n_q=64, n_kv=8, d=128, n=8, act="swiglu",
                       w_std=0.02, eps=1e-5),
    # the layer with every forward projection on per-tensor scaled E4M3
    # (bf16 storage, bf16 backward)
    "layer_fp8": dict(kind="layer", dtype="bf16", gemm_dtype="fp8", b=1,
                      s=8192, h=8192, h_ffn=28672, n_q=64, n_kv=8, d=128, n=8,
                      act="swiglu", w_std=0.02, eps=1e-5),
}

# Fixed sub-seed index of every tensor a workload draws.
_SUB = {"X": 1, "W1": 2, "b1": 3, "W2": 4, "b2": 5, "R": 6, "dOut": 7,
        "Wq": 8, "Wk": 9, "Wv": 10, "Wo": 11, "bo": 12, "g1": 13, "g2": 14}

TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


def workload(name, **overrides):
    """A copy of a named workload with some fields replaced (e.g. a smaller s)."""
    cfg = copy.deepcopy(WORKLOADS[name])
    cfg.update(overrides)
    cfg["name"] = name
    return cfg


def _normal(shape, std, seed, device, dtype, mean=0.0):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t.to(dtype)


def normal(shape, std, seed, device="cpu", dtype=torch.bfloat16, mean=0.0):
    """A seeded N(mean, std²) tensor rounded to ``dtype`` (the draw every
    workload tensor uses)."""
    return _normal(shape, std, seed, device, dtype, mean)


def _std(cfg, fan_in):
    w = cfg["w_std"]
    return fan_in ** -0.5 if w == "fan_in" else float(w)


def mlp_inputs(cfg, seed, device="cpu"):
    """X, W1, W2 (+ b1, b2, R, dOut) for an MLP workload, on ``device``."""
    T, h, f = cfg["b"] * cfg["s"], cfg["h"], cfg["h_ffn"]
    dt = TORCH_DTYPE[cfg["dtype"]]
    rows1 = 2 * f if cfg["act"] == "swiglu" else f
    out = {
        "X": _normal((T, h), 1.0, seed + _SUB["X"], device, dt),
        "W1": _normal((rows1, h), _std(cfg, h), seed + _SUB["W1"], device, dt),
        "W2": _normal((h, f), _std(cfg, f), seed + _SUB["W2"], device, dt),
        "dOut": _normal((T, h), 1.0, seed + _SUB["dOut"], device, dt),
        "b1": None, "b2": None, "R": None,
    }
    if cfg.get("b1"):
        out["b1"] = _normal((rows1,), 0.02, seed + _SUB["b1"], device, dt)
    if cfg.get("b2"):
        out["b2"] = _normal((h,), 0.02, seed + _SUB["b2"], device, dt)
    if cfg.get("residual") == "X":
        out["R"] = out["X"]
    elif cfg.get("residual") == "random":
        out["R"] = _normal((T, h), 1.0, seed + _SUB["R"], device, dt)
    return out


def attn_inputs(cfg, seed, device="cpu"):
    """X, Wq, Wk, Wv, Wo (+ bo, R, dOut) for an attention workload."""
    T, h, d = cfg["b"] * cfg["s"], cfg["h"], cfg["d"]
    nq, nkv = cfg["n_q"], cfg["n_kv"]
    dt = TORCH_DTYPE[cfg["dtype"]]
    out = {
        "X": _normal((T, h), 1.0, seed + _SUB["X"], device, dt),
        "Wq": _normal((nq * d, h), _std(cfg, h), seed + _SUB["Wq"], device, dt),
        "Wk": _normal((nkv * d, h), _std(cfg, h), seed + _SUB["Wk"], device,
                      dt),
        "Wv": _normal((nkv * d, h), _std(cfg, h), seed + _SUB["Wv"], device,
                      dt),
        "Wo": _normal((h, nq * d), _std(cfg, nq * d), seed + _SUB["Wo"],
                      device, dt),
        "dOut": _normal((T, h), 1.0, seed + _SUB["dOut"], device, dt),
        "bo": None, "R": None,
    }
    if cfg.get("bo"):
        out["bo"] = _normal((h,), 0.02, seed + _SUB["bo"], device, dt)
    if cfg.get("residual") == "X":
        out["R"] = out["X"]
    elif cfg.get("residual") == "random":
        out["R"] = _normal((T, h), 1.0, seed + _SUB["R"], device, dt)
    return out


def layer_inputs(cfg, seed, device="cpu"):
    """x, the layer's weights g1, Wq, Wk, Wv, Wo, g2, W1, W2, and dOut."""
    a = attn_inputs(dict(cfg, causal=True), seed, device)
    m = mlp_inputs(dict(cfg, residual=None, b1=False, b2=False, p=0.0), seed,
                   device)
    dt = TORCH_DTYPE[cfg["dtype"]]
    h = cfg["h"]
    return {
        "X": a["X"], "dOut": a["dOut"],
        "Wq": a["Wq"], "Wk": a["Wk"], "Wv": a["Wv"], "Wo": a["Wo"],
        "W1": m["W1"], "W2": m["W2"],
        "g1": _normal((h,), 0.02, seed + _SUB["g1"], device, dt, mean=1.0),
        "g2": _normal((h,), 0.02, seed + _SUB["g2"], device, dt, mean=1.0),
    }


def to_f64(t):
    """Exact float64 numpy copy of a (possibly bf16) tensor, or None."""
    if t is None:
        return None
    return t.detach().to("cpu", torch.float64).numpy()
