"""Pins for the fp64 backward oracle (``oracle.attention_backward``):

* torch autograd in float64 on the CPU, through an independent torch
  restatement of the forward (library cross-check), for every mask, ALiBi,
  softcap and GQA;
* central finite differences of L = sum(dO * O) through the (separately
  pinned) forward oracle, element by element on tiny inputs;
* invariants: the rows of dS sum to zero, so identical keys give dQ = 0; the
  key/value gradients of a GQA group are the sums over its query heads of
  the MHA gradients on repeated K/V.
"""
import numpy as np
import pytest
import torch

import oracle

RNG = np.random.default_rng(99)


def _rand(*shape):
    return RNG.standard_normal(shape)


def _torch_forward(q, k, v, scale, vis, score_mod=None, slopes=None, cap=None, grp=1):
    kk = k.repeat_interleave(grp, dim=1)
    vv = v.repeat_interleave(grp, dim=1)
    s = scale * torch.einsum("bhid,bhjd->bhij", q, kk)
    Lq, Lk = s.shape[-2:]
    if score_mod == "alibi":
        rel = torch.arange(Lk, dtype=torch.float64)[None, :] - torch.arange(Lq, dtype=torch.float64)[:, None]
        s = s + slopes[None, :, None, None] * rel
    elif score_mod == "softcap":
        s = cap * torch.tanh(s / cap)
    s = s.masked_fill(~vis, float("-inf"))
    return torch.softmax(s, dim=-1) @ vv


VARIANTS = [
    dict(),
    dict(mask="causal"),
    dict(mask="window", window=4),
    dict(mask="prefix_lm", prefix=5),
    dict(mask="document", doc_offsets=np.array([[0, 3, 7, 11], [0, 5, 6, 11]])),
    dict(mask="document", doc_offsets=np.array([[0, 3, 7, 11], [0, 5, 6, 11]]), doc_causal=True),
    dict(score_mod="alibi", mask="causal"),
    dict(score_mod="softcap", softcap=1.5),
]


@pytest.mark.parametrize("kw", VARIANTS, ids=lambda kw: "-".join(str(v) for v in kw.values()
                                                                 if isinstance(v, (str, int, float))) or "vanilla")
@pytest.mark.parametrize("grp", [1, 2])
def test_backward_matches_torch_autograd(kw, grp):
    B, Hkv, L, d = 2, 2, 11, 8
    Hq = Hkv * grp
    q, k, v, dout = _rand(B, Hq, L, d), _rand(B, Hkv, L, d), _rand(B, Hkv, L, d), _rand(B, Hq, L, d)
    slopes = np.array([0.5, 0.25, 0.125, 0.0625])[:Hq]
    okw = dict(kw)
    if kw.get("score_mod") == "alibi":
        okw["slopes"] = slopes
    dq, dk, dv = oracle.attention_backward(q, k, v, dout, scale=0.35, **okw)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    vis = torch.from_numpy(np.stack([oracle.visibility(kw.get("mask", "none"), L, L, window=kw.get("window"),
                                                       prefix=kw.get("prefix"),
                                                       offsets=None if "doc_offsets" not in kw else kw["doc_offsets"][b],
                                                       doc_causal=kw.get("doc_causal", False))
                                     for b in range(B)])[:, None])
    out = _torch_forward(tq, tk, tv, 0.35, vis, kw.get("score_mod"), torch.tensor(slopes), kw.get("softcap"), grp)
    out.backward(torch.tensor(dout))
    np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-12)


@pytest.mark.parametrize("kw", [dict(mask="causal"), dict(score_mod="softcap", softcap=0.9),
                                dict(score_mod="alibi", mask="window", window=3)])
def test_backward_finite_differences(kw):
    B, H, L, d = 1, 2, 6, 3
    q, k, v, dout = _rand(B, H, L, d), _rand(B, H, L, d), _rand(B, H, L, d), _rand(B, H, L, d)
    okw = dict(kw)
    if kw.get("score_mod") == "alibi":
        okw["slopes"] = np.array([0.7, 0.3])
    grads = oracle.attention_backward(q, k, v, dout, **okw)
    eps = 1e-6

    def loss(qq, kk, vv):
        o, _ = oracle.attention(qq, kk, vv, **okw)
        return float(np.sum(o * dout))

    for which, arr in enumerate((q, k, v)):
        for idx in [(0, 0, 0, 0), (0, 1, 3, 2), (0, 1, 5, 1), (0, 0, 2, 1)]:
            p, m = arr.copy(), arr.copy()
            p[idx] += eps
            m[idx] -= eps
            args_p = [q, k, v]
            args_m = [q, k, v]
            args_p[which], args_m[which] = p, m
            fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            assert grads[which][idx] == pytest.approx(fd, abs=1e-7), (which, idx)


def test_backward_identical_keys_give_zero_dq():
    B, H, L, d = 1, 2, 9, 4
    q, v, dout = _rand(B, H, L, d), _rand(B, H, L, d), _rand(B, H, L, d)
    k = np.broadcast_to(_rand(B, H, 1, d), (B, H, L, d)).copy()
    for kw in (dict(), dict(mask="causal"), dict(mask="prefix_lm", prefix=3)):
        dq, _, _ = oracle.attention_backward(q, k, v, dout, **kw)
        np.testing.assert_allclose(dq, 0.0, atol=1e-12)


def test_backward_gqa_sums_group_gradients():
    B, Hkv, grp, L, d = 1, 2, 3, 7, 4
    q, dout = _rand(B, Hkv * grp, L, d), _rand(B, Hkv * grp, L, d)
    k, v = _rand(B, Hkv, L, d), _rand(B, Hkv, L, d)
    dq, dk, dv = oracle.attention_backward(q, k, v, dout, mask="causal")
    kr, vr = np.repeat(k, grp, axis=1), np.repeat(v, grp, axis=1)
    dq2, dk2, dv2 = oracle.attention_backward(q, kr, vr, dout, mask="causal")
    np.testing.assert_allclose(dq, dq2, atol=1e-12)
    np.testing.assert_allclose(dk, dk2.reshape(B, Hkv, grp, L, d).sum(2), atol=1e-12)
    np.testing.assert_allclose(dv, dv2.reshape(B, Hkv, grp, L, d).sum(2), atol=1e-12)


# Differential attention backward: central finite differences of
# L = sum(dO * out) through the separately pinned forward oracle
# (oracle.diff_attention), for every one of the five inputs, causal and not;
# a dropped branch, a wrong sign of lambda or a missing dV term fails it.
@pytest.mark.parametrize("causal", [True, False])
def test_diff_backward_finite_differences(causal):
    B, H, L, d, dv, lam = 1, 2, 5, 3, 4, 0.6
    q1, k1, q2, k2 = (_rand(B, H, L, d) for _ in range(4))
    v, dout = _rand(B, H, L, dv), _rand(B, H, L, dv)
    grads = oracle.diff_attention_backward(q1, k1, q2, k2, v, dout, lam, causal=causal)
    eps = 1e-6

    def loss(*a):
        o, _, _ = oracle.diff_attention(*a, lam, causal=causal)
        return float(np.sum(o * dout))

    base = [q1, k1, q2, k2, v]
    for which in range(5):
        for idx in [(0, 0, 0, 0), (0, 1, 4, 2), (0, 1, 2, 1), (0, 0, 3, 0)]:
            p, m = [a.copy() for a in base], [a.copy() for a in base]
            p[which][idx] += eps
            m[which][idx] -= eps
            fd = (loss(*p) - loss(*m)) / (2 * eps)
            assert grads[which][idx] == pytest.approx(fd, abs=1e-7), (which, idx)


def test_diff_backward_lambda_zero_is_branch_one():
    """lambda = 0: the second branch gets no gradient and the rest is the
    plain attention backward of branch 1."""
    B, H, L, d, dv = 1, 2, 7, 4, 6
    q1, k1, q2, k2 = (_rand(B, H, L, d) for _ in range(4))
    v, dout = _rand(B, H, L, dv), _rand(B, H, L, dv)
    dq1, dk1, dq2, dk2, dvv = oracle.diff_attention_backward(q1, k1, q2, k2, v, dout, 0.0, causal=True)
    rq, rk, rv = oracle.attention_backward(q1, k1, v, dout, mask="causal")
    assert np.array_equal(dq2, np.zeros_like(dq2)) and np.array_equal(dk2, np.zeros_like(dk2))
    np.testing.assert_allclose(dq1, rq, rtol=0, atol=1e-13)
    np.testing.assert_allclose(dk1, rk, rtol=0, atol=1e-13)
    np.testing.assert_allclose(dvv, rv, rtol=0, atol=1e-13)
