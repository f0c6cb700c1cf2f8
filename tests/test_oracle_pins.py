"""Pins for the fp64 oracle: things other than the oracle itself that fix
what it must return.

* closed forms (uniform scores give LSE = log #visible and the mean of the
  visible V rows; hand-worked two-key softcap / ALiBi / gate examples;
  one-hot bias entries in the Evoformer pick out one V row),
* invariants (rows of P sum to 1, shift invariance, causal row 0 = V[0]),
* special cases that reduce to vanilla or causal attention,
* a library cross-check against torch's scaled_dot_product_attention in
  float64 on the CPU,
* a scalar brute-force loop on L <= 16,
* the pages' claim that the online single-pass softmax equals the two-pass
  stable softmax (Flashlight technical summary, gist.science, Methodology:
  "Semantic Fusion with Algebraic Transformation").

Each plausible slip in the oracle -- a dropped scale, a wrong ALiBi sign,
softcap applied before the scale, an off-by-one window or prefix, a wrong
document boundary, a wrong GQA head map, a transposed pair bias, a wrong
sign on lambda -- fails at least one test here.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from flashattention_attn_fwd_gb300 import synth
from tests._brute import brute_row

RNG = np.random.default_rng(1234)


def _rand(*shape):
    return RNG.standard_normal(shape)


def _mask_kwargs(mask, L):
    if mask == "window":
        return dict(window=5)
    if mask == "prefix_lm":
        return dict(prefix=4)
    if mask == "document":
        return dict(doc_offsets=np.array([[0, 3, 4, L]]))
    return {}


def _visible_count(mask, i, L, kw, doc_causal=False):
    """Hand-derived number of keys visible to query i (Lq == Lk == L)."""
    if mask == "none":
        return L
    if mask == "causal":
        return i + 1
    if mask == "window":
        return min(i + 1, kw["window"])
    if mask == "prefix_lm":
        return max(i + 1, kw["prefix"])
    if mask == "document":
        off = list(kw["doc_offsets"][0])
        for a, b in zip(off[:-1], off[1:]):
            if a <= i < b:
                return (i - a + 1) if doc_causal else (b - a)
    raise ValueError(mask)


@pytest.mark.parametrize("mask", oracle.MASKS)
def test_uniform_scores_closed_form(mask):
    """q = 0 makes every score 0: LSE_i = log(#visible keys) and out_i is the
    plain mean of the visible V rows.  Pins every mask's key count."""
    L, d = 11, 4
    q = np.zeros((1, 1, L, d))
    k = _rand(1, 1, L, d)
    v = _rand(1, 1, L, 3)
    kw = _mask_kwargs(mask, L)
    out, lse = oracle.attention(q, k, v, mask=mask, **kw)
    vis = oracle.visibility(mask, L, L, window=kw.get("window"), prefix=kw.get("prefix"),
                            offsets=kw.get("doc_offsets", [None])[0])
    for i in range(L):
        n = _visible_count(mask, i, L, kw)
        assert vis[i].sum() == n
        assert lse[0, 0, i] == pytest.approx(math.log(n), abs=1e-13)
        np.testing.assert_allclose(out[0, 0, i], v[0, 0][vis[i]].mean(axis=0), atol=1e-13)


def test_document_causal_counts():
    L = 11
    kw = dict(doc_offsets=np.array([[0, 3, 4, L]]))
    q = np.zeros((1, 1, L, 2))
    _, lse = oracle.attention(q, _rand(1, 1, L, 2), _rand(1, 1, L, 2), mask="document",
                              doc_causal=True, **kw)
    for i in range(L):
        assert lse[0, 0, i] == pytest.approx(math.log(_visible_count("document", i, L, kw, True)))


@pytest.mark.parametrize("mask", oracle.MASKS)
def test_identical_keys_give_mean_of_visible_values(mask):
    L, d = 9, 5
    q = _rand(1, 2, L, d)
    k = np.repeat(_rand(1, 2, 1, d), L, axis=2)
    v = _rand(1, 2, L, 6)
    kw = _mask_kwargs(mask, L)
    out, _ = oracle.attention(q, k, v, mask=mask, **kw)
    vis = oracle.visibility(mask, L, L, window=kw.get("window"), prefix=kw.get("prefix"),
                            offsets=kw.get("doc_offsets", [None])[0])
    for h in range(2):
        for i in range(L):
            np.testing.assert_allclose(out[0, h, i], v[0, h][vis[i]].mean(axis=0), atol=1e-12)


def test_rows_of_p_sum_to_one_and_causal_row0():
    q, k, v = _rand(2, 3, 13, 8), _rand(2, 3, 13, 8), _rand(2, 3, 13, 8)
    for mask in oracle.MASKS:
        kw = _mask_kwargs(mask, 13)
        if mask == "document":
            kw = dict(doc_offsets=np.array([[0, 3, 4, 13], [0, 7, 8, 13]]))
        _, _, P = oracle.attention(q, k, v, mask=mask, return_probs=True, **kw)
        np.testing.assert_allclose(P.sum(-1), 1.0, atol=1e-13)
        assert (P >= 0).all()
    out, _ = oracle.attention(q, k, v, mask="causal")
    np.testing.assert_allclose(out[:, :, 0], v[:, :, 0], atol=1e-15)


def test_scale_is_applied_to_logits():
    """Two keys, d = 1: scores are scale*q*k, checked by hand."""
    q = np.array([[[[2.0]]]])
    k = np.array([[[[1.0], [-0.5]]]])
    v = np.array([[[[1.0], [0.0]]]])
    for scale in (1.0, 0.25):
        out, lse = oracle.attention(q, k, v, scale=scale)
        t0, t1 = scale * 2.0, scale * -1.0
        p0 = math.exp(t0) / (math.exp(t0) + math.exp(t1))
        assert out[0, 0, 0, 0] == pytest.approx(p0, abs=1e-15)
        assert lse[0, 0, 0] == pytest.approx(math.log(math.exp(t0) + math.exp(t1)), abs=1e-14)
    out, _ = oracle.attention(np.ones((1, 1, 1, 4)), np.ones((1, 1, 2, 4)), v)
    assert out[0, 0, 0, 0] == pytest.approx(0.5)  # equal scores: default scale irrelevant


def test_softcap_closed_form_after_scaling():
    """softcap acts on the *scaled* logit: t = cap*tanh(scale*q.k / cap)."""
    q = np.array([[[[3.0]]]])
    k = np.array([[[[4.0], [-1.0]]]])
    v = np.array([[[[1.0], [0.0]]]])
    scale, cap = 0.5, 1.5
    out, lse = oracle.attention(q, k, v, scale=scale, score_mod="softcap", softcap=cap)
    t0 = cap * math.tanh(scale * 12.0 / cap)
    t1 = cap * math.tanh(scale * -3.0 / cap)
    assert out[0, 0, 0, 0] == pytest.approx(math.exp(t0) / (math.exp(t0) + math.exp(t1)), abs=1e-15)
    assert lse[0, 0, 0] == pytest.approx(math.log(math.exp(t0) + math.exp(t1)), abs=1e-14)


def test_alibi_sign_closed_form():
    """q = 0: t_ij = m (j - i); later keys gain weight for m > 0."""
    L, m = 3, 0.7
    q = np.zeros((1, 1, L, 2))
    k = _rand(1, 1, L, 2)
    v = np.eye(L)[None, None]
    out, lse = oracle.attention(q, k, v, score_mod="alibi", slopes=[m])
    for i in range(L):
        w = [math.exp(m * (j - i)) for j in range(L)]
        z = sum(w)
        np.testing.assert_allclose(out[0, 0, i], [x / z for x in w], atol=1e-15)
        assert lse[0, 0, i] == pytest.approx(math.log(z), abs=1e-14)


def test_special_cases_reduce_to_vanilla_or_causal():
    B, H, L, d = 2, 2, 10, 6
    q, k, v = _rand(B, H, L, d), _rand(B, H, L, d), _rand(B, H, L, d)
    van = oracle.attention(q, k, v)
    cau = oracle.attention(q, k, v, mask="causal")

    def same(a, b, tol=1e-12):
        np.testing.assert_allclose(a[0], b[0], atol=tol)
        np.testing.assert_allclose(a[1], b[1], atol=tol)

    same(oracle.attention(q, k, v, score_mod="alibi", slopes=[0.0, 0.0]), van)
    same(oracle.attention(q, k, v, score_mod="softcap", softcap=1e30), van)
    same(oracle.attention(q, k, v, mask="window", window=L), cau)
    same(oracle.attention(q, k, v, mask="window", window=10 * L), cau)
    same(oracle.attention(q, k, v, mask="prefix_lm", prefix=0), cau)
    same(oracle.attention(q, k, v, mask="prefix_lm", prefix=1), cau)
    same(oracle.attention(q, k, v, mask="prefix_lm", prefix=L), van)
    one = np.array([[0, L], [0, L]])
    same(oracle.attention(q, k, v, mask="document", doc_offsets=one), van)
    same(oracle.attention(q, k, v, mask="document", doc_offsets=one, doc_causal=True), cau)
    # window 1 = each query sees only itself
    out, lse = oracle.attention(q, k, v, mask="window", window=1)
    np.testing.assert_allclose(out, v, atol=1e-15)
    np.testing.assert_allclose(lse, np.einsum("bhid,bhid->bhi", q, k) / math.sqrt(d), atol=1e-13)


def test_gqa_equals_mha_on_repeated_kv():
    B, Hq, Hkv, L, d = 2, 8, 2, 9, 4
    q, k, v = _rand(B, Hq, L, d), _rand(B, Hkv, L, d), _rand(B, Hkv, L, 5)
    kr, vr = np.repeat(k, Hq // Hkv, axis=1), np.repeat(v, Hq // Hkv, axis=1)
    slopes = 2.0 ** (-np.arange(1, Hq + 1))
    for kw in (dict(), dict(mask="causal"), dict(score_mod="alibi", slopes=slopes)):
        a = oracle.attention(q, k, v, **kw)
        b = oracle.attention(q, kr, vr, **kw)
        np.testing.assert_allclose(a[0], b[0], atol=1e-14)
        np.testing.assert_allclose(a[1], b[1], atol=1e-14)
    # and head h of the group really reads kv head h // (Hq/Hkv)
    out, _ = oracle.attention(q, k, v)
    for h in range(Hq):
        ref, _ = oracle.attention(q[:, h:h + 1], k[:, h // 4:h // 4 + 1], v[:, h // 4:h // 4 + 1])
        np.testing.assert_allclose(out[:, h], ref[:, 0], atol=1e-14)


def _sdpa(q, k, v, attn_mask=None, gqa=False):
    return F.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v),
        attn_mask=None if attn_mask is None else torch.from_numpy(attn_mask),
        enable_gqa=gqa).numpy()


@pytest.mark.parametrize("mask", oracle.MASKS)
def test_library_crosscheck_sdpa_masks(mask):
    B, Hq, Hkv, L, d = 2, 4, 2, 37, 16
    q, k, v = _rand(B, Hq, L, d), _rand(B, Hkv, L, d), _rand(B, Hkv, L, 8)
    kw = dict(window=7) if mask == "window" else dict(prefix=9) if mask == "prefix_lm" else {}
    if mask == "document":
        offs = np.array([[0, 5, 6, 20, L], [0, 1, 30, 31, L]])
        kw = dict(doc_offsets=offs)
        bm = np.stack([oracle.visibility("document", L, L, offsets=o) for o in offs])[:, None]
    else:
        bm = np.broadcast_to(oracle.visibility(mask, L, L, **kw), (B, 1, L, L)).copy()
    out, _ = oracle.attention(q, k, v, mask=mask, **kw)
    ref = _sdpa(q, k, v, attn_mask=bm, gqa=True)
    np.testing.assert_allclose(out, ref, atol=1e-12)


def test_library_crosscheck_sdpa_alibi():
    B, H, L, d = 1, 4, 29, 8
    q, k, v = _rand(B, H, L, d), _rand(B, H, L, d), _rand(B, H, L, d)
    slopes = synth.alibi_slopes(H).double().numpy()
    i, j = np.arange(L)[:, None], np.arange(L)[None, :]
    bias = (slopes[:, None, None] * (j - i)[None])[None]
    out, _ = oracle.attention(q, k, v, score_mod="alibi", slopes=slopes)
    np.testing.assert_allclose(out, _sdpa(q, k, v, attn_mask=bias), atol=1e-12)
    # slopes 2^(-8h/H), h = 1..H
    np.testing.assert_allclose(slopes, [2.0 ** (-8.0 * h / H) for h in range(1, H + 1)], rtol=1e-7)


def test_shift_invariance():
    """Adding c to every score of a row leaves O unchanged, shifts LSE by c."""
    B, Ns, H, Nr, d = 1, 2, 2, 7, 4
    q, k, v, g = (_rand(B, Ns, H, Nr, d) for _ in range(4))
    pb, mb = _rand(B, H, Nr, Nr), np.zeros((B, Ns, Nr))
    o1, l1 = oracle.evoformer_gated_attention(q, k, v, pb, mb, g)
    o2, l2 = oracle.evoformer_gated_attention(q, k, v, pb + 3.25, mb, g)
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(l2 - l1, 3.25, atol=1e-12)


def test_evoformer_reduces_to_vanilla():
    B, Ns, H, Nr, d = 1, 3, 2, 9, 8
    q, k, v = (_rand(B, Ns, H, Nr, d) for _ in range(3))
    gate = np.full((B, Ns, H, Nr, d), 40.0)  # sigmoid(40) == 1 in fp64
    out, lse = oracle.evoformer_gated_attention(q, k, v, np.zeros((B, H, Nr, Nr)),
                                                np.zeros((B, Ns, Nr)), gate)
    ref, rl = oracle.attention(q.reshape(B * Ns, H, Nr, d), k.reshape(B * Ns, H, Nr, d),
                               v.reshape(B * Ns, H, Nr, d))
    np.testing.assert_allclose(out.reshape(ref.shape), ref, atol=1e-14)
    np.testing.assert_allclose(lse.reshape(rl.shape), rl, atol=1e-14)


def test_evoformer_bias_indexing_one_hot():
    """A large pair_bias[h, i0, j0] makes query i0 of head h copy V row j0
    (for every MSA row); a mask bias that hides all but key j1 of MSA row s
    makes every query of that row copy V row j1.  Gate scales elementwise."""
    B, Ns, H, Nr, d = 1, 3, 2, 6, 4
    q, k, v, g = (_rand(B, Ns, H, Nr, d) for _ in range(4))
    pb = np.zeros((B, H, Nr, Nr))
    pb[0, 1, 2, 4] = 80.0
    mb = np.zeros((B, Ns, Nr))
    mb[0, 2, :] = -1e9
    mb[0, 2, 3] = 0.0
    out, _ = oracle.evoformer_gated_attention(q, k, v, pb, mb, g)
    sig = 1 / (1 + np.exp(-g))
    for s in (0, 1):
        np.testing.assert_allclose(out[0, s, 1, 2], sig[0, s, 1, 2] * v[0, s, 1, 4], atol=1e-12)
    for h in range(H):
        for i in range(Nr):
            np.testing.assert_allclose(out[0, 2, h, i], sig[0, 2, h, i] * v[0, 2, h, 3], atol=1e-12)


def test_evoformer_gate_closed_form():
    B, Ns, H, Nr, d = 1, 1, 1, 4, 3
    q, k, g = (_rand(B, Ns, H, Nr, d) for _ in range(3))
    v = np.broadcast_to(np.array([1.5, -2.0, 0.25]), (B, Ns, H, Nr, d)).copy()
    out, _ = oracle.evoformer_gated_attention(q, k, v, _rand(B, H, Nr, Nr), np.zeros((B, Ns, Nr)), g)
    for i in range(Nr):
        for c in range(d):
            assert out[0, 0, 0, i, c] == pytest.approx(v[0, 0, 0, 0, c] / (1 + math.exp(-g[0, 0, 0, i, c])))


def test_diff_attention_lambda():
    B, H, L = 1, 2, 12
    q1, k1, q2, k2 = (_rand(B, H, L, 8) for _ in range(4))
    v = _rand(B, H, L, 16)
    base, bl = oracle.attention(q1, k1, v, mask="causal", scale=0.125)
    out, l1, l2 = oracle.diff_attention(q1, k1, q2, k2, v, 0.0, scale=0.125)
    np.testing.assert_allclose(out, base, atol=1e-14)
    np.testing.assert_allclose(l1, bl, atol=1e-14)
    # q2 = 0: branch 2 is the causal running mean of v, subtracted with weight lambda
    out, _, l2 = oracle.diff_attention(q1, k1, np.zeros_like(q2), k2, v, 0.8, scale=0.125)
    run_mean = np.cumsum(v, axis=2) / np.arange(1, L + 1)[None, None, :, None]
    np.testing.assert_allclose(out, base - 0.8 * run_mean, atol=1e-13)
    np.testing.assert_allclose(l2, np.broadcast_to(np.log(np.arange(1, L + 1)), l2.shape), atol=1e-13)
    # identical branches with lambda = 1 cancel
    out, _, _ = oracle.diff_attention(q1, k1, q1, k1, v, 1.0, scale=0.125)
    np.testing.assert_allclose(out, 0.0, atol=1e-14)


def test_fully_masked_row_gives_zero_and_neg_inf():
    t = np.array([[-np.inf, -np.inf], [0.0, 1.0]])
    P, lse = oracle.softmax_rows(t)
    assert (P[0] == 0).all() and lse[0] == -np.inf
    assert P[1].sum() == pytest.approx(1.0)


VARIANTS = [
    dict(),
    dict(mask="causal"),
    dict(mask="window", window=3),
    dict(mask="prefix_lm", prefix=5),
    dict(mask="document", doc_offsets=np.array([[0, 2, 9, 13]])),
    dict(mask="document", doc_offsets=np.array([[0, 2, 9, 13]]), doc_causal=True),
    dict(score_mod="alibi", slopes=[0.5, 0.125]),
    dict(score_mod="softcap", softcap=2.0),
    dict(mask="causal", score_mod="softcap", softcap=1.0),
]


@pytest.mark.parametrize("kw", VARIANTS, ids=lambda kw: "-".join(f"{a}" for a in kw.values() if isinstance(a, (str, int, float))) or "vanilla")
def test_brute_force_small(kw):
    B, H, L, d = 1, 2, 13, 5
    q, k, v = _rand(B, H, L, d), _rand(B, H, L, d), _rand(B, H, L, 3)
    out, lse = oracle.attention(q, k, v, **kw)
    mk = {}
    if "window" in kw:
        mk["window"] = kw["window"]
    if "prefix" in kw:
        mk["prefix"] = kw["prefix"]
    if "doc_offsets" in kw:
        mk["offsets"] = list(kw["doc_offsets"][0])
        mk["doc_causal"] = kw.get("doc_causal", False)
    for h in range(H):
        for i in range(L):
            o, l = brute_row(q[0, h, i].tolist(), k[0, h].tolist(), v[0, h].tolist(), i,
                             1 / math.sqrt(d), mask=kw.get("mask", "none"),
                             score_mod=kw.get("score_mod", "none"),
                             slope=(kw.get("slopes") or [0, 0])[h], cap=kw.get("softcap"), **mk)
            np.testing.assert_allclose(out[0, h, i], o, atol=1e-12)
            assert lse[0, h, i] == pytest.approx(l, abs=1e-12)


def test_brute_force_evoformer():
    B, Ns, H, Nr, d = 1, 2, 2, 7, 4
    q, k, v, g = (_rand(B, Ns, H, Nr, d) for _ in range(4))
    pb, mb = _rand(B, H, Nr, Nr), np.where(RNG.random((B, Ns, Nr)) < 0.7, 0.0, -1e9)
    mb[..., 0] = 0.0
    out, lse = oracle.evoformer_gated_attention(q, k, v, pb, mb, g)
    for s in range(Ns):
        for h in range(H):
            for i in range(Nr):
                bias = [pb[0, h, i, j] + mb[0, s, j] for j in range(Nr)]
                o, l = brute_row(q[0, s, h, i].tolist(), k[0, s, h].tolist(), v[0, s, h].tolist(),
                                 i, 1 / math.sqrt(d), bias_row=bias)
                sig = [1 / (1 + math.exp(-x)) for x in g[0, s, h, i]]
                np.testing.assert_allclose(out[0, s, h, i], [a * b for a, b in zip(sig, o)], atol=1e-12)
                assert lse[0, s, h, i] == pytest.approx(l, abs=1e-12)


def test_decode_reduces_to_prefix_attention():
    """One new row with the whole cache visible is vanilla attention over
    the first kv_len keys; Lq rows with the causal mask and kv_len == Lq is
    causal self-attention; ALiBi is measured from the row's own position."""
    B, Hq, Hkv, Lq, Lmax, d = 3, 4, 2, 1, 20, 8
    q, k, v = _rand(B, Hq, Lq, d), _rand(B, Hkv, Lmax, d), _rand(B, Hkv, Lmax, d)
    lens = np.array([20, 7, 1])
    out, lse = oracle.decode_attention(q, k, v, lens)
    for b in range(B):
        n = lens[b]
        ro, rl = oracle.attention(q[b:b + 1], k[b:b + 1, :, :n], v[b:b + 1, :, :n])
        np.testing.assert_allclose(out[b:b + 1], ro, atol=1e-13)
        np.testing.assert_allclose(lse[b:b + 1], rl, atol=1e-13)
    Lq = 5
    q2 = _rand(B, Hq, Lq, d)
    out, lse = oracle.decode_attention(q2, k[:, :, :Lq], v[:, :, :Lq], np.full(B, Lq), causal=True)
    ro, rl = oracle.attention(q2, k[:, :, :Lq], v[:, :, :Lq], mask="causal")
    np.testing.assert_allclose(out, ro, atol=1e-13)
    np.testing.assert_allclose(lse, rl, atol=1e-13)


def test_decode_causal_offset_and_sdpa_crosscheck():
    """Bottom-right causal alignment against torch SDPA (float64) with an
    explicit boolean mask, plus the q = 0 closed form: the last row sees
    kv_len keys, row i sees kv_len - Lq + i + 1."""
    B, Hq, Hkv, Lq, Lmax, d = 2, 4, 2, 3, 16, 8
    q, k, v = _rand(B, Hq, Lq, d), _rand(B, Hkv, Lmax, d), _rand(B, Hkv, Lmax, d)
    lens = np.array([16, 9])
    out, lse = oracle.decode_attention(q, k, v, lens, causal=True)
    for b in range(B):
        n = lens[b]
        i = np.arange(Lq)[:, None]
        j = np.arange(Lmax)[None, :]
        m = (j < n) & (j <= n - Lq + i)
        ref = _sdpa(q[b:b + 1], np.repeat(k[b:b + 1], 2, axis=1), np.repeat(v[b:b + 1], 2, axis=1), attn_mask=m)
        np.testing.assert_allclose(out[b:b + 1], ref, atol=1e-12)
    out0, lse0 = oracle.decode_attention(np.zeros_like(q), k, v, lens, causal=True)
    for b in range(B):
        for i in range(Lq):
            cnt = lens[b] - Lq + i + 1
            np.testing.assert_allclose(lse0[b, :, i], math.log(cnt), atol=1e-12)
            np.testing.assert_allclose(out0[b, 0, i], v[b, 0, :cnt].mean(0), atol=1e-12)


def test_brute_force_decode():
    B, Hq, Hkv, Lq, Lmax, d = 2, 2, 1, 2, 9, 4
    q, k, v = _rand(B, Hq, Lq, d), _rand(B, Hkv, Lmax, d), _rand(B, Hkv, Lmax, d)
    lens = np.array([9, 4])
    slopes = np.array([0.5, 0.125])
    for kw in (dict(), dict(causal=True), dict(score_mod="alibi", slopes=slopes, causal=True),
               dict(score_mod="softcap", softcap=1.5)):
        out, lse = oracle.decode_attention(q, k, v, lens, scale=0.4, **kw)
        for b in range(B):
            n = int(lens[b])
            for h in range(Hq):
                for i in range(Lq):
                    p = n - Lq + i
                    K = k[b, 0, :n].tolist()
                    V = v[b, 0, :n].tolist()
                    # brute_row's causal is j <= row index: pass the position
                    mk = dict(mask="causal") if kw.get("causal") else {}
                    sm = {}
                    if kw.get("score_mod") == "alibi":
                        sm = dict(score_mod="alibi", slope=float(slopes[h]))
                    elif kw.get("score_mod") == "softcap":
                        sm = dict(score_mod="softcap", cap=1.5)
                    o, l = brute_row(q[b, h, i].tolist(), K, V, p, 0.4, **mk, **sm)
                    np.testing.assert_allclose(out[b, h, i], o, atol=1e-12)
                    assert lse[b, h, i] == pytest.approx(l, abs=1e-12)


def test_evoformer_col_is_row_form_on_transposed_msa():
    """Column-wise attention over MSA rows = the (separately pinned) row-wise
    form on the MSA with its two axes swapped, with zero pair bias and the
    column mask as the row mask."""
    B, Ns, H, Nr, d = 2, 7, 2, 5, 4
    q, k, v, g = (_rand(B, Ns, H, Nr, d) for _ in range(4))
    mb = np.where(RNG.random((B, Nr, Ns)) < 0.7, 0.0, -1e9)
    mb[..., 0] = 0.0
    out, lse = oracle.evoformer_col_gated_attention(q, k, v, mb, g)
    tr = lambda x: np.ascontiguousarray(np.swapaxes(x, 1, 3))  # noqa: E731
    ro, rl = oracle.evoformer_gated_attention(tr(q), tr(k), tr(v), np.zeros((B, H, Ns, Ns)), mb, tr(g))
    np.testing.assert_allclose(out, tr(ro), atol=1e-13)
    np.testing.assert_allclose(lse, np.swapaxes(rl, 1, 2), atol=1e-13)


def test_evoformer_col_closed_forms():
    """q = 0: every visible MSA row weighs the same, so out is sigmoid(gate)
    times the mean of the visible V rows of that column and lse = log
    #visible; a mask keeping one MSA row s0 copies V[s0]."""
    B, Ns, H, Nr, d = 1, 6, 2, 3, 4
    k, v, g = (_rand(B, Ns, H, Nr, d) for _ in range(3))
    q = np.zeros((B, Ns, H, Nr, d))
    mb = np.zeros((B, Nr, Ns))
    mb[0, 1, [0, 2, 5]] = -1e9
    mb[0, 2, :] = -1e9
    mb[0, 2, 4] = 0.0
    out, lse = oracle.evoformer_col_gated_attention(q, k, v, mb, g)
    sig = 1 / (1 + np.exp(-g))
    for h in range(H):
        for s in range(Ns):
            np.testing.assert_allclose(out[0, s, h, 0], sig[0, s, h, 0] * v[0, :, h, 0].mean(0), atol=1e-12)
            np.testing.assert_allclose(out[0, s, h, 1], sig[0, s, h, 1] * v[0, [1, 3, 4], h, 1].mean(0), atol=1e-12)
            np.testing.assert_allclose(out[0, s, h, 2], sig[0, s, h, 2] * v[0, 4, h, 2], atol=1e-12)
    np.testing.assert_allclose(lse[0, :, 0], math.log(Ns), atol=1e-12)
    np.testing.assert_allclose(lse[0, :, 1], math.log(3), atol=1e-12)


def test_brute_force_evoformer_col():
    B, Ns, H, Nr, d = 1, 7, 2, 3, 4
    q, k, v, g = (_rand(B, Ns, H, Nr, d) for _ in range(4))
    mb = np.where(RNG.random((B, Nr, Ns)) < 0.7, 0.0, -1e9)
    mb[..., 0] = 0.0
    out, lse = oracle.evoformer_col_gated_attention(q, k, v, mb, g, scale=0.3)
    for h in range(H):
        for r in range(Nr):
            K = [k[0, s, h, r].tolist() for s in range(Ns)]
            V = [v[0, s, h, r].tolist() for s in range(Ns)]
            for s in range(Ns):
                o, l = brute_row(q[0, s, h, r].tolist(), K, V, s, 0.3, bias_row=mb[0, r].tolist())
                sig = [1 / (1 + math.exp(-x)) for x in g[0, s, h, r]]
                np.testing.assert_allclose(out[0, s, h, r], [a * b for a, b in zip(sig, o)], atol=1e-12)
                assert lse[0, h, r, s] == pytest.approx(l, abs=1e-12)


def test_evoformer_col_rows_match_full():
    e = synth.evo_col_inputs(1, 9, 5, 2, d=8, seed=3)
    out, lse = oracle.evoformer_col_gated_attention(*e)
    rows = [(0, 0, 0, 0), (0, 8, 1, 4), (0, 3, 1, 2)]
    ro, rl = oracle.evoformer_col_rows(*e, rows=rows)
    for n, (b, s, h, r) in enumerate(rows):
        np.testing.assert_allclose(ro[n], out[b, s, h, r], atol=1e-13)
        assert rl[n] == pytest.approx(lse[b, h, r, s], abs=1e-13)


@pytest.mark.parametrize("kw", VARIANTS[:-1], ids=lambda kw: "-".join(f"{a}" for a in kw.values() if isinstance(a, (str, int, float))) or "vanilla")
@pytest.mark.parametrize("block", [4, 16])
def test_online_equals_two_pass(kw, block):
    B, H, L, d = 1, 2, 13, 5
    q, k, v = _rand(B, H, L, d) * 3, _rand(B, H, L, d), _rand(B, H, L, 3)
    a = oracle.attention(q, k, v, **kw)
    b = oracle.online_attention(q, k, v, block=block, **kw)
    np.testing.assert_allclose(a[0], b[0], atol=1e-12)
    np.testing.assert_allclose(a[1], b[1], atol=1e-12)


def test_rows_match_full():
    q, k, v = synth.attn_inputs(2, 4, 2, 40, 8, seed=3)
    offs = synth.doc_offsets(2, 40, 4, seed=3)
    slopes = synth.alibi_slopes(4)
    rows = [(0, 0, 0), (1, 3, 39), (0, 2, 17), (1, 1, 5)]
    for kw in (dict(), dict(mask="causal"), dict(mask="window", window=6),
               dict(mask="prefix_lm", prefix=11), dict(mask="document", doc_offsets=offs),
               dict(mask="document", doc_offsets=offs, doc_causal=True),
               dict(score_mod="alibi", slopes=slopes), dict(score_mod="softcap", softcap=3.0)):
        full_o, full_l = oracle.attention(q, k, v, **kw)
        ro, rl = oracle.attention_rows(q, k, v, rows, **kw)
        for n, (b, h, i) in enumerate(rows):
            np.testing.assert_allclose(ro[n], full_o[b, h, i], atol=1e-13)
            assert rl[n] == pytest.approx(full_l[b, h, i], abs=1e-13)
    q1, k1, q2, k2, vv = synth.diff_inputs(1, 2, 20, d=8, dv=16, seed=1)
    fo, f1, f2 = oracle.diff_attention(q1, k1, q2, k2, vv, 0.8)
    ro, r1, r2 = oracle.diff_attention_rows(q1, k1, q2, k2, vv, 0.8, [(0, 1, 7)])
    np.testing.assert_allclose(ro[0], fo[0, 1, 7], atol=1e-13)
    e = synth.evo_inputs(1, 3, 10, 2, d=4, seed=2)
    fo, fl = oracle.evoformer_gated_attention(*e)
    ro, rl = oracle.evoformer_rows(*e, rows=[(0, 2, 1, 9)])
    np.testing.assert_allclose(ro[0], fo[0, 2, 1, 9], atol=1e-13)
    assert rl[0] == pytest.approx(fl[0, 2, 1, 9])


def test_synth_inputs_are_seeded_and_shaped():
    a = synth.attn_inputs(1, 2, 1, 5, 4, seed=7)
    b = synth.attn_inputs(1, 2, 1, 5, 4, seed=7)
    for x, y in zip(a, b):
        assert torch.equal(x, y) and x.dtype == torch.bfloat16
    offs = synth.doc_offsets(3, 100, 8, seed=1)
    assert offs.shape == (3, 9) and (offs[:, 0] == 0).all() and (offs[:, -1] == 100).all()
    assert (offs[:, 1:] > offs[:, :-1]).all()
    e = synth.evo_inputs(1, 4, 16, 2, seed=0, p_keep=0.05)
    assert ((e[4] == 0).sum(-1) >= 1).all()


def test_golden_fixture_reproduces():
    """The stored fixture (written by tests/golden/make_golden.py from the
    oracle) still matches the oracle on the same seeded inputs."""
    import json
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "causal_b1h2l256d64_seed0.json")
    fx = json.load(open(path))
    q, k, v = synth.attn_inputs(1, 2, 2, 256, 64, seed=0)
    ro, rl = oracle.attention_rows(q, k, v, [tuple(r) for r in fx["rows"]], mask="causal")
    np.testing.assert_allclose(ro, np.array(fx["out"]), atol=1e-12)
    np.testing.assert_allclose(rl, np.array(fx["lse"]), atol=1e-12)
    # causal row 0 is V[0] exactly
    np.testing.assert_allclose(fx["out"][0], v[0, 0, 0].double().numpy(), atol=0)
