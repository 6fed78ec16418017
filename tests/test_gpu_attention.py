"""GPU parity of the head-sharded GQA attention block against the oracle."""

import numpy as np
import pytest
import torch

import oracle
from megatron_tensor_transformer_gate_gb300 import inputs as I
from megatron_tensor_transformer_gate_gb300.blocks import TPAttention
from _parity import check, check_fro

pytestmark = pytest.mark.gpu


def run_case(tp, cfg, mode, seed):
    b, s, h = cfg["b"], cfg["s"], cfg["h"]
    nq, nkv, d, n = cfg["n_q"], cfg["n_kv"], cfg["d"], cfg["n"]
    causal = cfg.get("causal", True)
    x = I.attn_inputs(cfg, seed, "cpu")
    dv = {k: (v.cuda() if v is not None else None) for k, v in x.items()}
    a = TPAttention(b, s, h, nq, nkv, d, n, causal=causal, mode=mode)
    out = a.forward(dv["X"], dv["Wq"], dv["Wk"], dv["Wv"], dv["Wo"],
                    bo=dv["bo"], R=dv["R"])
    g = a.backward(dv["dOut"], dv["X"], dv["Wq"], dv["Wk"], dv["Wv"],
                   dv["Wo"], want_dbo=x["bo"] is not None)
    tp.device_status()
    f = {k: I.to_f64(v) for k, v in x.items()}
    kw = dict(b=b, s=s, n_q=nq, n_kv=nkv, d=d, causal=causal)
    fo = oracle.attention_forward(f["X"], f["Wq"], f["Wk"], f["Wv"], f["Wo"],
                                  bo=f["bo"], R=f["R"], **kw)
    go = oracle.attention_backward(f["dOut"], f["X"], f["Wq"], f["Wk"],
                                   f["Wv"], f["Wo"], fo, **kw)
    check(out, fo["Out"], "Out")
    for k in ("dX", "dWq", "dWk", "dWv", "dWo"):
        check(g[k], go[k], k)
    if "dbo" in g:
        check(g["dbo"], go["dbo"], "dbo")


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("causal", [True, False])
def test_ragged_small(tp, mode, causal):
    # s not a multiple of the 128/64 blocks; 2 batches; GQA group 4
    cfg = I.workload("attn_gqa_bf16", b=2, s=200, h=512, n_q=8, n_kv=2, n=2,
                     causal=causal, bo=True, residual="random",
                     w_std="fan_in")
    run_case(tp, cfg, mode, 31)


@pytest.mark.parametrize("mode", [0, 1])
def test_mqa_single_kv_per_rank(tp, mode):
    cfg = I.workload("attn_gqa_bf16", b=1, s=300, h=1024, n_q=8, n_kv=4, n=4,
                     w_std="fan_in")
    run_case(tp, cfg, mode, 32)


@pytest.mark.parametrize("mode", [0, 1])
def test_gqa_workload(tp, mode):
    run_case(tp, I.workload("attn_gqa_bf16"), mode, 20260004)


def test_fp16_overflow_is_reported(tp):
    # inputs scaled so that Q = X·Wqᵀ exceeds the fp16 range: the library
    # must report TP_ERR_RANGE through the device status word (no fault)
    cfg = I.workload("attn_gqa_bf16", b=1, s=64, h=256, n_q=2, n_kv=1, n=1,
                     w_std="fan_in")
    x = I.attn_inputs(cfg, 33, "cuda")
    X = (x["X"].float() * 1e5).to(x["X"].dtype)
    a = TPAttention(1, 64, 256, 2, 1, 128, 1)
    a.forward(X, x["Wq"], x["Wk"], x["Wv"], x["Wo"])
    with pytest.raises(tp.TPError) as e:
        tp.device_status()
    assert e.value.code == 9
    tp.device_status()          # the word was cleared by the read


def test_gqa_layer_widths(tp):
    # the attention block of the layer workload (h 8192, 64 q / 8 kv heads,
    # n 8) at s = 512 on its own seeded inputs, both bounds
    cfg = I.workload("attn_gqa_bf16", b=1, s=512, h=8192, n_q=64, n_kv=8,
                     n=8)
    run_case(tp, cfg, 0, 20260005)


def test_overlapped_reduction_attention_workload(tp):
    # the attention workload (T 4096) with the out-projection g and the input
    # gradient f reduced band by band: against the oracle, and bit-identical
    # to the materialised mode
    cfg = I.workload("attn_gqa_bf16")
    run_case(tp, cfg, tp.OVERLAP, 20260004)
    x = I.attn_inputs(cfg, 20260004, "cuda")
    res = []
    for mode in (tp.MATERIALISED, tp.OVERLAP):
        a = TPAttention(cfg["b"], cfg["s"], cfg["h"], cfg["n_q"], cfg["n_kv"],
                        cfg["d"], cfg["n"], mode=mode)
        out = a.forward(x["X"], x["Wq"], x["Wk"], x["Wv"], x["Wo"])
        g = a.backward(x["dOut"], x["X"], x["Wq"], x["Wk"], x["Wv"], x["Wo"])
        tp.device_status()
        res.append([out.clone(), g["dX"].clone()])
    for u, v in zip(*res):
        assert u.equal(v)


@pytest.mark.parametrize("causal", [True, False])
def test_backward_in_passes_is_bit_identical(tp, causal):
    # a dS budget below one (batch, kv head) pair's tiles runs the backward
    # in one pass per pair (4 here): smaller scratch, identical results
    cfg = I.workload("attn_gqa_bf16", b=2, s=200, h=512, n_q=8, n_kv=2, n=2,
                     causal=causal, w_std="fan_in")
    x = I.attn_inputs(cfg, 34, "cuda")
    res, scratch = [], []
    for budget in (0, 1):
        prev = tp.attn_set_ds_budget(budget)
        try:
            a = TPAttention(cfg["b"], cfg["s"], cfg["h"], cfg["n_q"],
                            cfg["n_kv"], cfg["d"], cfg["n"], causal=causal)
            scratch.append(tp.attn_bwd_scratch_bytes(a.desc))
            out = a.forward(x["X"], x["Wq"], x["Wk"], x["Wv"], x["Wo"])
            g = a.backward(x["dOut"], x["X"], x["Wq"], x["Wk"], x["Wv"],
                           x["Wo"])
            tp.device_status()
            res.append([out.clone()] + [g[k].clone() for k in
                                        ("dX", "dWq", "dWk", "dWv", "dWo")])
        finally:
            tp.attn_set_ds_budget(prev)
    assert scratch[1] < scratch[0]
    for u, v in zip(*res):
        assert u.equal(v)


@pytest.mark.parametrize("n_q,n_kv,n", [(8, 8, 2), (32, 2, 2)])
def test_group_size_extremes(tp, n_q, n_kv, n):
    # plain multi-head attention (one q head per kv head) and a wide GQA
    # group of 16 q heads per kv head, ragged s
    cfg = I.workload("attn_gqa_bf16", b=1, s=260, h=1024, n_q=n_q, n_kv=n_kv,
                     n=n, w_std="fan_in")
    run_case(tp, cfg, 0, 38)


@pytest.mark.parametrize("n_q,n_kv", [(4, 2), (4, 4)])
@pytest.mark.parametrize("causal", [True, False])
def test_sequences_shorter_than_a_block(tp, n_q, n_kv, causal):
    # s = 77 < 128: one partial key block per sequence, three sequences; the
    # forward's output rows past the end are clipped on store.  GQA group 2
    # pairs two heads in a CTA; group 1 pairs query blocks, and the second
    # one is past the end in every CTA
    cfg = I.workload("attn_gqa_bf16", b=3, s=77, h=512, n_q=n_q, n_kv=n_kv,
                     n=2, causal=causal, w_std="fan_in")
    run_case(tp, cfg, 0, 44)


@pytest.mark.parametrize("b,s", [(1, 384), (2, 500)])
@pytest.mark.parametrize("causal", [True, False])
def test_odd_group_size(tp, b, s, causal):
    # three q heads per kv head on each rank: the forward then puts two
    # consecutive query blocks of one head in a CTA instead of two heads of
    # a group; s = 384 leaves the last CTA's second block past the end
    # (three blocks), s = 500 fills both with a ragged tail (four blocks),
    # over two sequences
    cfg = I.workload("attn_gqa_bf16", b=b, s=s, h=1024, n_q=12, n_kv=4, n=2,
                     causal=causal, w_std="fan_in")
    run_case(tp, cfg, 0, 41)


@pytest.mark.parametrize("causal", [True, False])
def test_single_token_sequences(tp, causal):
    # s = 1: each query attends only to its own key (softmax weight 1), so
    # the block reduces to the V and output projections and dQ, dWq are
    # exactly 0.  The kernels form dS = P·(dP − D) with D taken from the
    # stored bf16 O, so dQ is rounding noise instead: it is held against the
    # scale of dWv (the same product with dV for dQ); everything else
    # against the oracle as usual
    b, s, h, nq, nkv, d, n = 2, 1, 512, 4, 2, 128, 2
    cfg = I.workload("attn_gqa_bf16", b=b, s=s, h=h, n_q=nq, n_kv=nkv, n=n,
                     causal=causal, w_std="fan_in")
    x = I.attn_inputs(cfg, 40, "cpu")
    dv = {k: (v.cuda() if v is not None else None) for k, v in x.items()}
    a = TPAttention(b, s, h, nq, nkv, d, n, causal=causal)
    out = a.forward(dv["X"], dv["Wq"], dv["Wk"], dv["Wv"], dv["Wo"])
    g = a.backward(dv["dOut"], dv["X"], dv["Wq"], dv["Wk"], dv["Wv"],
                   dv["Wo"])
    tp.device_status()
    f = {k: I.to_f64(v) for k, v in x.items()}
    kw = dict(b=b, s=s, n_q=nq, n_kv=nkv, d=d, causal=causal)
    fo = oracle.attention_forward(f["X"], f["Wq"], f["Wk"], f["Wv"], f["Wo"],
                                  **kw)
    go = oracle.attention_backward(f["dOut"], f["X"], f["Wq"], f["Wk"],
                                   f["Wv"], f["Wo"], fo, **kw)
    assert np.abs(go["dWq"]).max() == 0.0
    check(out, fo["Out"], "Out")
    for k in ("dX", "dWv", "dWo"):
        check(g[k], go[k], k)
    scale = np.linalg.norm(go["dWv"])
    for k in ("dWq", "dWk"):
        err = np.linalg.norm(g[k].double().cpu().numpy() - go[k])
        assert err <= 1e-2 * scale, (k, err / scale)


def _rescaled_rows(f, cfg):
    """Rows whose running reference max the forward kernel moves: the first
    key block's row max is the reference, and a later block's row max above
    it by more than 2^12 in exp2 units (12 / (scale·log2 e) in raw scores)
    replaces it."""
    b, s, d = cfg["b"], cfg["s"], cfg["d"]
    nq, nkv = cfg["n_q"], cfg["n_kv"]
    thr = 12.0 / ((1.0 / np.sqrt(d)) * np.log2(np.e))
    X = f["X"].reshape(b, s, -1)
    count = 0
    for bi in range(b):
        for j in range(nq):
            q = X[bi] @ f["Wq"][j * d:(j + 1) * d].T
            kv = j // (nq // nkv)
            k = X[bi] @ f["Wk"][kv * d:(kv + 1) * d].T
            S = q @ k.T
            if cfg.get("causal", True):
                S = np.where(np.tril(np.ones((s, s), dtype=bool)), S, -np.inf)
            for r in range(s):
                m_ref = None
                for k0 in range(0, s, 128):
                    bm = S[r, k0:k0 + 128].max()
                    if bm == -np.inf:
                        break
                    if m_ref is None:
                        m_ref = bm
                    elif bm > m_ref + thr:
                        m_ref = bm
                        count += 1
                        break
    return count


@pytest.mark.parametrize("causal", [True, False])
def test_growing_scores_rescale_the_output(tp, causal):
    # inputs whose rows grow along the sequence, so that a query's scores
    # against later key blocks exceed the first block's maximum by far more
    # than the kernel's rescale threshold: the accumulated output and row
    # sum are rescaled, possibly several times per row.  The output is held
    # to both bounds.  Such rows' softmax is nearly one-hot, where
    # dS = P·(dP − D) cancels exactly in the oracle but leaves rounding
    # noise in the kernels (D from the stored bf16 O), so the gradients are
    # held to the Frobenius bound
    b, s, h, nq, nkv, d, n = 1, 512, 512, 8, 2, 128, 2
    cfg = I.workload("attn_gqa_bf16", b=b, s=s, h=h, n_q=nq, n_kv=nkv, n=n,
                     causal=causal, w_std="fan_in")
    x = I.attn_inputs(cfg, 42, "cpu")
    grow = 1.0 + np.arange(s) / 128.0
    x["X"] = (x["X"].float() *
              torch.from_numpy(np.tile(grow, b)).float()[:, None]).to(
                  x["X"].dtype)
    f = {k: I.to_f64(v) for k, v in x.items()}
    assert _rescaled_rows(f, cfg) > s * nq // 4   # the path is exercised
    dv = {k: (v.cuda() if v is not None else None) for k, v in x.items()}
    a = TPAttention(b, s, h, nq, nkv, d, n, causal=causal)
    out = a.forward(dv["X"], dv["Wq"], dv["Wk"], dv["Wv"], dv["Wo"])
    g = a.backward(dv["dOut"], dv["X"], dv["Wq"], dv["Wk"], dv["Wv"],
                   dv["Wo"])
    tp.device_status()
    kw = dict(b=b, s=s, n_q=nq, n_kv=nkv, d=d, causal=causal)
    fo = oracle.attention_forward(f["X"], f["Wq"], f["Wk"], f["Wv"], f["Wo"],
                                  **kw)
    go = oracle.attention_backward(f["dOut"], f["X"], f["Wq"], f["Wk"],
                                   f["Wv"], f["Wo"], fo, **kw)
    check(out, fo["Out"], "Out")
    for k in ("dX", "dWq", "dWk", "dWv", "dWo"):
        check_fro(g[k], go[k], k)


def _rescale_events(f, cfg, thr_log2=12.0):
    """(q head, query row, key block) of every new reference max under the
    forward kernel's rule: the first key block's row max is the reference,
    and a later block's row max above it by more than 2^12 in exp2 units
    replaces it."""
    b, s, d = cfg["b"], cfg["s"], cfg["d"]
    nq, nkv = cfg["n_q"], cfg["n_kv"]
    thr = thr_log2 / ((1.0 / np.sqrt(d)) * np.log2(np.e))
    X = f["X"].reshape(b, s, -1)
    ev = set()
    for bi in range(b):
        for j in range(nq):
            kv = j // (nq // nkv)
            S = (X[bi] @ f["Wq"][j * d:(j + 1) * d].T) @ (
                X[bi] @ f["Wk"][kv * d:(kv + 1) * d].T).T
            if cfg.get("causal", True):
                S = np.where(np.tril(np.ones((s, s), dtype=bool)), S, -np.inf)
            for r in range(s):
                m_ref = None
                for k0 in range(0, s, 128):
                    bm = S[r, k0:k0 + 128].max()
                    if bm == -np.inf:
                        break
                    if m_ref is None:
                        m_ref = bm
                    elif bm > m_ref + thr:
                        m_ref = bm
                        ev.add((j, r, k0 // 128))
    return ev


@pytest.mark.parametrize("causal", [True, False])
def test_rescale_of_a_few_rows_of_one_tile(tp, causal):
    # The forward accumulates Oᵀ (column = query), so a row's rescale is
    # carried out on its column by all four warps of the tile, for the
    # 32-column chunk of the warp quarter that flagged it.  Here a marker
    # feature makes the scores of a few chosen query rows jump at one later
    # key block (rows 296-301: quarter 1 of the third query tile, and row
    # 400: quarter 0 of the fourth), while every other row keeps its first
    # block's reference: a rescale applied to the wrong chunk, or skipped,
    # shows in those rows' outputs.  Feature 0 of every q head comes only
    # from input column 0 (set on the marked query rows) and feature 0 of
    # every kv head only from input column 1 (set on keys 200-205 and 390),
    # so the marked rows' scores against the marked keys gain
    # (2·10)² / √d (log2 units: 51, far above the threshold of 12) and no
    # other score changes.  Gradients are held to the Frobenius bound (nearly one-hot
    # rows, as for the growing scores).
    b, s, h, nq, nkv, d, n = 1, 512, 512, 8, 2, 128, 2
    cfg = I.workload("attn_gqa_bf16", b=b, s=s, h=h, n_q=nq, n_kv=nkv, n=n,
                     causal=causal, w_std="fan_in")
    x = I.attn_inputs(cfg, 7, "cpu")
    X = x["X"].float()
    Wq, Wk = x["Wq"].float(), x["Wk"].float()
    marked_q = list(range(296, 302)) + [400]
    marked_k = list(range(200, 206)) + [390]
    X[:, 0] = 0.0
    X[:, 1] = 0.0
    X[marked_q, 0] = 10.0
    X[marked_k, 1] = 10.0
    Wq[:, :2] = 0.0
    Wk[:, :2] = 0.0
    Wq[torch.arange(nq) * d, :] = 0.0
    Wk[torch.arange(nkv) * d, :] = 0.0
    Wq[torch.arange(nq) * d, 0] = 2.0
    Wk[torch.arange(nkv) * d, 1] = 2.0
    x["X"], x["Wq"], x["Wk"] = (X.to(x["X"].dtype), Wq.to(x["Wq"].dtype),
                                Wk.to(x["Wk"].dtype))
    f = {k: I.to_f64(v) for k, v in x.items()}
    ev = _rescale_events(f, cfg)
    rows = {r for (_, r, _) in ev}
    assert set(marked_q) <= rows                  # the marked rows rescale
    assert len(rows - set(marked_q)) <= 8         # few others do
    assert {(r // 128, (r % 128) // 32) for r in marked_q} == {(2, 1), (3, 0)}
    dv = {k: (v.cuda() if v is not None else None) for k, v in x.items()}
    a = TPAttention(b, s, h, nq, nkv, d, n, causal=causal)
    out = a.forward(dv["X"], dv["Wq"], dv["Wk"], dv["Wv"], dv["Wo"])
    g = a.backward(dv["dOut"], dv["X"], dv["Wq"], dv["Wk"], dv["Wv"],
                   dv["Wo"])
    tp.device_status()
    kw = dict(b=b, s=s, n_q=nq, n_kv=nkv, d=d, causal=causal)
    fo = oracle.attention_forward(f["X"], f["Wq"], f["Wk"], f["Wv"], f["Wo"],
                                  **kw)
    go = oracle.attention_backward(f["dOut"], f["X"], f["Wq"], f["Wk"],
                                   f["Wv"], f["Wo"], fo, **kw)
    check(out, fo["Out"], "Out")
    # the marked rows themselves, row by row, against the oracle
    o = out.float().cpu().numpy()
    ref = fo["Out"]
    for r in marked_q:
        err = np.abs(o[r] - ref[r]).max() / np.sqrt(np.mean(ref[r] ** 2))
        assert err <= 3e-2, (r, err)
    for k in ("dX", "dWq", "dWk", "dWv", "dWo"):
        check_fro(g[k], go[k], k)


@pytest.mark.parametrize("causal", [True, False])
def test_growing_scores_odd_group(tp, causal):
    # Three q heads per kv head: the forward pairs two consecutive query
    # blocks of one head in a CTA, so under the causal mask the second tile
    # goes on alone (one N=128 output product per block) after the first has
    # ended, and s = 640 (five blocks) leaves the last CTA's second tile past
    # the end.  Rows growing by 1 + t/256 make many rows take new reference
    # maxima, some of them in the blocks where the second tile runs alone
    # (CPU replay of the rule), with softmax rows less peaked than at
    # 1 + t/128, whose nearly one-hot rows put dWq's rounding noise (D from
    # the bf16 O) at the Frobenius bound.  Output to both bounds, gradients
    # to the Frobenius bound.
    b, s, h, nq, nkv, d, n = 1, 640, 1024, 12, 4, 128, 2
    cfg = I.workload("attn_gqa_bf16", b=b, s=s, h=h, n_q=nq, n_kv=nkv, n=n,
                     causal=causal, w_std="fan_in")
    x = I.attn_inputs(cfg, 43, "cpu")
    grow = 1.0 + np.arange(s) / 256.0
    x["X"] = (x["X"].float() *
              torch.from_numpy(np.tile(grow, b)).float()[:, None]).to(
                  x["X"].dtype)
    f = {k: I.to_f64(v) for k, v in x.items()}
    ev = _rescale_events(f, cfg)
    assert len({(j, r) for (j, r, _) in ev}) > s * nq // 4
    if causal:
        alone = [e for e in ev if (e[1] // 128) % 2 == 1 and e[2] == e[1] // 128]
        assert len(alone) > 100
    dv = {k: (v.cuda() if v is not None else None) for k, v in x.items()}
    a = TPAttention(b, s, h, nq, nkv, d, n, causal=causal)
    out = a.forward(dv["X"], dv["Wq"], dv["Wk"], dv["Wv"], dv["Wo"])
    g = a.backward(dv["dOut"], dv["X"], dv["Wq"], dv["Wk"], dv["Wv"],
                   dv["Wo"])
    tp.device_status()
    kw = dict(b=b, s=s, n_q=nq, n_kv=nkv, d=d, causal=causal)
    fo = oracle.attention_forward(f["X"], f["Wq"], f["Wk"], f["Wv"], f["Wo"],
                                  **kw)
    go = oracle.attention_backward(f["dOut"], f["X"], f["Wq"], f["Wk"],
                                   f["Wv"], f["Wo"], fo, **kw)
    check(out, fo["Out"], "Out")
    for k in ("dX", "dWq", "dWk", "dWv", "dWo"):
        check_fro(g[k], go[k], k)

