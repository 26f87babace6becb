"""MoE router select and expert FFN against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from gemm_decode_prefill_gb300 import synth
from gpu_helpers import TOL_GEMV, TOL_ROUTER_W, assert_within, dev, host, moe_bound

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qmv():
    from gemm_decode_prefill_gb300 import qmv as m
    return m


def _check_select(qmv, logits, k, renorm, sgw=None, x=None, sg_logit=None):
    kw = {}
    if sgw is not None:
        kw = dict(sg_w=dev(sgw), x=dev(x))
    elif sg_logit is not None:
        kw = dict(sg_logit=dev(np.array([sg_logit], np.float32)))
    sel, w = qmv.moe_select_topk(dev(logits), k, renorm, **kw)
    sel, w = host(sel), host(w)
    sel_ref, w_ref = oracle.select(logits, k, renorm, sgw=sgw, x=x, sg_logit=sg_logit)
    assert sel.tolist() == sel_ref.tolist()
    np.testing.assert_allclose(w.astype(np.float64), w_ref, rtol=TOL_ROUTER_W, atol=0)


@pytest.mark.parametrize("n", [1, 2, 7, 32, 128, 257, 1024])
def test_select_random_logits(qmv, n):
    g = synth.rng(70 + n)
    logits = g.standard_normal(n).astype(np.float32)
    for k in sorted({1, min(2, n), min(8, n), n}):
        for renorm in (False, True):
            _check_select(qmv, logits, k, renorm)


def test_select_ties_pick_lowest_index(qmv):
    g = synth.rng(80)
    for n in (5, 64, 128, 300):
        logits = g.integers(0, 3, size=n).astype(np.float32)
        for k in (1, 3, 8, n):
            if k <= n:
                _check_select(qmv, logits, k, True)
    z = np.array([(-1) ** i * 0.0 for i in range(16)], np.float32)   # +0 / -0 compare equal
    _check_select(qmv, z, 5, False)


def test_select_shared_gate(qmv):
    m = synth.moe_inputs(n_exp=128, hidden=2048, inter=16, seed=81)
    _check_select(qmv, m.logits, 8, True, sgw=m.sgw, x=m.x)
    _check_select(qmv, m.logits, 8, False, sg_logit=-0.75)
    big = (m.sgw * 40).astype(np.float32)  # a large gate logit
    _check_select(qmv, m.logits, 8, True, sgw=big, x=m.x)


def test_select_rejects_bad_arguments(qmv):
    with pytest.raises(qmv.QmvError, match="INVALID_ARG"):
        qmv.moe_select_topk(dev(np.zeros(8, np.float32)), 9, True)
    with pytest.raises(qmv.QmvError, match="INVALID_ARG"):
        qmv.moe_select_topk(dev(np.zeros(1025, np.float32)), 2, True)


def _pack_moe(qmv, m):
    return (qmv.qmv_pack_q8row(dev(m.gq), dev(m.grs)), qmv.qmv_pack_q8row(dev(m.uq), dev(m.urs)),
            qmv.qmv_pack_q8row(dev(m.dq), dev(m.drs)))


def _run_step(qmv, m, k, renorm):
    gate, up, down = _pack_moe(qmv, m)
    sel, w = qmv.moe_select_topk(dev(m.logits), k, renorm, sg_w=dev(m.sgw), x=dev(m.x))
    out = qmv.moe_ffn_q8row(gate, up, down, sel, w, dev(m.x))
    return host(sel), host(w), host(out)


@pytest.mark.parametrize("n_exp,hidden,inter,k", [(6, 64, 48, 1), (10, 128, 96, 3), (128, 2048, 768, 8)])
def test_moe_step_matches_oracle(qmv, n_exp, hidden, inter, k):
    m = synth.moe_inputs(n_exp, hidden, inter, seed=90 + n_exp)
    sel, w, out = _run_step(qmv, m, k, True)
    sel_ref, w_ref = oracle.select(m.logits, k, True, sgw=m.sgw, x=m.x)
    assert sel.tolist() == sel_ref.tolist()
    np.testing.assert_allclose(w.astype(np.float64), w_ref, rtol=TOL_ROUTER_W, atol=0)
    out_ref, parts = oracle.moe_ffn(m.gq, m.grs, m.uq, m.urs, m.dq, m.drs, sel_ref, w_ref, m.x,
                                    with_parts=True)
    bound = moe_bound(m, sel_ref, w_ref, parts)
    assert_within(out, out_ref, bound, 1.0, f"moe {n_exp}x{hidden}x{inter} k={k}")


def test_moe_ffn_given_selection_matches_oracle(qmv):
    """The FFN stage alone, fed the same (sel, w) on both sides."""
    m = synth.moe_inputs(12, 256, 128, seed=95)
    gate, up, down = _pack_moe(qmv, m)
    sel = np.array([11, 0, 5, 12, 5], np.int32)   # repeats and the shared block
    w = np.array([0.5, -0.25, 1.5, 0.75, 0.125], np.float32)
    out = host(qmv.moe_ffn_q8row(gate, up, down, dev(sel), dev(w), dev(m.x)))
    out_ref, parts = oracle.moe_ffn(m.gq, m.grs, m.uq, m.urs, m.dq, m.drs, sel, w.astype(np.float64), m.x,
                                    with_parts=True)
    assert_within(out, out_ref, moe_bound(m, sel, w, parts), 1.0, "moe ffn given selection")


def test_moe_bad_expert_sets_device_status(qmv):
    m = synth.moe_inputs(4, 64, 32, seed=96)
    gate, up, down = _pack_moe(qmv, m)
    qmv.qmv_check()
    sel = dev(np.array([1, 9], np.int32))   # 9 is out of range (5 experts)
    w = dev(np.array([1.0, 1.0], np.float32))
    qmv.moe_ffn_q8row(gate, up, down, sel, w, dev(m.x))
    with pytest.raises(qmv.QmvError, match="DEVICE_STATUS"):
        qmv.qmv_check()
    assert qmv.qmv_check() == 0   # cleared


# (n_exp, hidden, inter, top_k, shared, renorm): the rank path (n_exp <= 256)
# and the argmax-rounds path (n_exp > 256), with and without a shared expert,
# with a given shared-gate logit, with and without renormalisation
FUSED_CASES = [(128, 2048, 768, 8, "sgw", True), (10, 128, 96, 3, "sgw", False), (300, 256, 64, 6, "logit", True),
               (64, 512, 128, 4, None, True), (7, 64, 48, 7, "sgw", True)]


@pytest.mark.parametrize("n_exp,hidden,inter,k,shared,renorm", FUSED_CASES)
def test_moe_step_fused_matches_separate_and_oracle(qmv, n_exp, hidden, inter, k, shared, renorm):
    m = synth.moe_inputs(n_exp, hidden, inter, seed=200 + n_exp + k)
    gate, up, down = _pack_moe(qmv, m)
    kw, okw = {}, {}
    if shared == "sgw":
        kw = dict(sg_w=dev(m.sgw))
        okw = dict(sgw=m.sgw, x=m.x)
    elif shared == "logit":
        kw = dict(sg_logit=dev(np.array([0.3], np.float32)))
        okw = dict(sg_logit=0.3)
    sel_f, w_f, out_f = qmv.moe_step_q8row(dev(m.logits), k, renorm, gate, up, down, dev(m.x), **kw)
    sel_s, w_s = qmv.moe_select_topk(dev(m.logits), k, renorm, x=dev(m.x) if shared == "sgw" else None, **kw)
    out_s = qmv.moe_ffn_q8row(gate, up, down, sel_s, w_s, dev(m.x))
    sel_f, w_f, out_f, sel_s, w_s, out_s = (host(t) for t in (sel_f, w_f, out_f, sel_s, w_s, out_s))
    assert np.array_equal(sel_f, sel_s) and np.array_equal(w_f, w_s)
    assert np.array_equal(out_f, out_s)
    sel_ref, w_ref = oracle.select(m.logits, k, renorm, **okw)
    assert sel_f.tolist() == sel_ref.tolist()
    np.testing.assert_allclose(w_f.astype(np.float64), w_ref, rtol=TOL_ROUTER_W, atol=0)
    out_ref, parts = oracle.moe_ffn(m.gq, m.grs, m.uq, m.urs, m.dq, m.drs, sel_ref, w_ref, m.x, with_parts=True)
    assert_within(out_f, out_ref, moe_bound(m, sel_ref, w_ref, parts), 1.0, "fused moe step")


def test_moe_step_rejects_too_few_experts(qmv):
    m = synth.moe_inputs(8, 64, 32, seed=97)   # stacks of 9 experts (8 routed + the shared one)
    gate, up, down = _pack_moe(qmv, m)
    logits = dev(np.zeros(9, np.float32))      # a router over 9 experts needs 10 with the shared one
    with pytest.raises(qmv.QmvError, match="INVALID_ARG"):
        qmv.moe_step_q8row(logits, 2, True, gate, up, down, dev(m.x), sg_w=dev(m.sgw))


# Shapes too wide for the staged FFN kernels, one per register-streaming
# fallback: the down projection of 9 slots x 2560 columns (2 x 9 x 10 KB of
# codes per CTA is over the 96 KB budget); gate/up rows of 12800 columns (x
# does not fit the 48 KB activation staging); gate/up rows of 9216 columns
# (x fits, but not three row groups of both matrices).
FALLBACK_CASES = [(8, 2048, 2560, 8), (2, 12800, 64, 1), (2, 9216, 64, 1)]


@pytest.mark.parametrize("n_exp,hidden,inter,k", FALLBACK_CASES)
def test_moe_step_register_fallbacks(qmv, n_exp, hidden, inter, k):
    m = synth.moe_inputs(n_exp, hidden, inter, seed=300 + n_exp + hidden)
    gate, up, down = _pack_moe(qmv, m)
    sel, w, out = qmv.moe_step_q8row(dev(m.logits), k, True, gate, up, down, dev(m.x), sg_w=dev(m.sgw))
    sel, w, out = host(sel), host(w), host(out)
    sel_ref, w_ref = oracle.select(m.logits, k, True, sgw=m.sgw, x=m.x)
    assert sel.tolist() == sel_ref.tolist()
    np.testing.assert_allclose(w.astype(np.float64), w_ref, rtol=TOL_ROUTER_W, atol=0)
    out_ref, parts = oracle.moe_ffn(m.gq, m.grs, m.uq, m.urs, m.dq, m.drs, sel_ref, w_ref, m.x, with_parts=True)
    assert_within(out, out_ref, moe_bound(m, sel_ref, w_ref, parts), 1.0, f"moe fallback {hidden}x{inter}")
