"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
the same seeded bf16 inputs.

Bar (per output tensor): max-abs error <= 2e-2, relative L2 error <= 1e-2,
LSE max-abs error <= 1e-3.  Small shapes are compared element by element;
the full-size workloads are compared on sampled query rows, each computed by
the oracle from the full K/V.
"""
import numpy as np
import pytest
import torch

import oracle
from flashattention_attn_fwd_gb300 import (FlattnError, attn_fwd, diffattn_fwd, evoformer_col_gated_attn_fwd,
                                           evoformer_gated_attn_fwd, synth, sync_status)
from flashattention_attn_fwd_gb300._lib import FL_DEBUG_KEY_SPLIT, FL_DEBUG_SKIP_KV_LOAD, FL_ERR_TIMEOUT

pytestmark = pytest.mark.gpu

ATOL, RTOL, LSE_ATOL = 2e-2, 1e-2, 1e-3
DEV = "cuda"


def _np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def check(out, ref, lse=None, ref_lse=None, atol=ATOL, rtol=RTOL, lse_atol=LSE_ATOL):
    g = _np(out)
    assert g.shape == ref.shape
    assert np.isfinite(g).all()
    err = np.abs(g - ref)
    mae = float(err.max()) if err.size else 0.0
    rel = float(np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-30))
    assert mae <= atol and rel <= rtol, f"max-abs {mae:.3e} rel-L2 {rel:.3e}"
    if lse is not None:
        gl = _np(lse)
        fin = np.isfinite(ref_lse)
        assert (np.isfinite(gl) == fin).all()
        lerr = float(np.abs(gl[fin] - ref_lse[fin]).max()) if fin.any() else 0.0
        assert lerr <= lse_atol, f"lse max-abs {lerr:.3e}"


def _gpu(*ts):
    return [t.to(DEV) for t in ts]


def _oracle_kw(kw, offs=None, slopes=None):
    o = {}
    for a in ("mask", "window", "prefix", "doc_causal", "score_mod", "softcap", "scale"):
        if a in kw:
            o[a] = kw[a]
    if offs is not None:
        o["doc_offsets"] = offs
    if slopes is not None:
        o["slopes"] = slopes
    return o


def run_attn(B, Hq, Hkv, L, d, seed=0, n_docs=None, dv=None, **kw):
    q, k, v = synth.attn_inputs(B, Hq, Hkv, L, d, dv=dv, seed=seed)
    offs = synth.doc_offsets(B, L, n_docs, seed=seed) if n_docs else None
    slopes = synth.alibi_slopes(Hq) if kw.get("score_mod") == "alibi" else None
    gkw = dict(kw)
    if offs is not None:
        gkw["doc_offsets"] = offs.to(DEV)
    if slopes is not None:
        gkw["alibi_slopes"] = slopes.to(DEV)
    out, lse = attn_fwd(*_gpu(q, k, v), **gkw)
    sync_status()
    return (q, k, v, offs, slopes), out, lse


SMALL = [
    # (B, Hq, Hkv, L, d, n_docs, kwargs)
    (1, 2, 2, 256, 64, None, dict(mask="causal")),
    (1, 2, 2, 256, 64, None, dict()),
    (2, 3, 3, 1, 64, None, dict()),
    (1, 2, 2, 17, 64, None, dict(mask="causal")),
    (1, 2, 2, 129, 64, None, dict()),
    (2, 2, 2, 255, 64, None, dict(mask="causal")),
    (1, 3, 3, 300, 64, None, dict(mask="causal")),
    (1, 2, 2, 384, 64, None, dict(mask="causal")),
    (1, 2, 2, 200, 32, None, dict(mask="causal")),
    (1, 2, 2, 200, 128, None, dict(mask="causal")),
    (1, 2, 2, 300, 32, None, dict()),
    (1, 2, 2, 300, 128, None, dict()),
    (1, 2, 2, 300, 64, None, dict(mask="window", window=37)),
    (1, 2, 2, 700, 64, None, dict(mask="window", window=256)),
    (1, 2, 2, 300, 64, None, dict(mask="window", window=1)),
    (1, 2, 2, 300, 64, None, dict(mask="prefix_lm", prefix=100)),
    (1, 2, 2, 600, 64, None, dict(mask="prefix_lm", prefix=300)),
    (1, 2, 2, 300, 64, None, dict(mask="prefix_lm", prefix=0)),
    (1, 2, 2, 300, 64, None, dict(mask="prefix_lm", prefix=300)),
    (2, 2, 2, 500, 64, 4, dict(mask="document")),
    (2, 2, 2, 500, 64, 4, dict(mask="document", doc_causal=True)),
    (1, 2, 2, 300, 64, 1, dict(mask="document")),
    (1, 4, 4, 300, 64, None, dict(score_mod="alibi")),
    (1, 4, 4, 300, 64, None, dict(score_mod="alibi", mask="causal")),
    (1, 2, 2, 300, 64, None, dict(score_mod="softcap", softcap=30.0)),
    (1, 2, 2, 300, 64, None, dict(score_mod="softcap", softcap=2.0, mask="causal")),
    (2, 8, 2, 300, 64, None, dict()),
    (2, 8, 2, 300, 64, None, dict(mask="causal")),
    (1, 6, 2, 300, 64, None, dict(mask="causal")),
    (1, 3, 1, 257, 64, None, dict()),
    (2, 8, 2, 520, 64, 5, dict(mask="document", doc_causal=True)),
    (1, 8, 2, 520, 64, None, dict(mask="prefix_lm", prefix=130, score_mod="softcap", softcap=10.0)),
    (1, 2, 2, 300, 64, None, dict(scale=0.3, mask="causal")),
]


def _id(c):
    B, Hq, Hkv, L, d, nd, kw = c
    tag = "-".join(f"{k}{v}" for k, v in kw.items())
    return f"B{B}H{Hq}x{Hkv}L{L}d{d}" + (f"docs{nd}" if nd else "") + (f"-{tag}" if tag else "")


@pytest.mark.parametrize("case", SMALL, ids=_id)
def test_attn_small_elementwise(case):
    B, Hq, Hkv, L, d, nd, kw = case
    (q, k, v, offs, slopes), out, lse = run_attn(B, Hq, Hkv, L, d, seed=L + d, n_docs=nd, **kw)
    ro, rl = oracle.attention(q, k, v, **_oracle_kw(kw, offs, slopes))
    check(out, ro, lse, rl)


DV_CASES = [
    # (B, Hq, Hkv, L, d, dv, kwargs): value head dim different from the query/key one
    (1, 2, 2, 300, 64, 128, dict(mask="causal")),
    (2, 8, 2, 300, 64, 128, dict(mask="causal")),
    (1, 2, 2, 300, 64, 128, dict(score_mod="alibi")),
    (1, 2, 2, 200, 32, 64, dict(mask="causal")),
    (1, 4, 2, 200, 32, 128, dict()),
    (1, 2, 2, 200, 128, 64, dict(mask="window", window=70)),
    (1, 2, 2, 300, 64, 32, dict(score_mod="softcap", softcap=5.0)),
    (1, 2, 2, 260, 128, 32, dict(mask="prefix_lm", prefix=50)),
]


@pytest.mark.parametrize("case", DV_CASES, ids=lambda c: f"B{c[0]}H{c[1]}x{c[2]}L{c[3]}d{c[4]}dv{c[5]}-" +
                         "-".join(f"{k}{v}" for k, v in c[6].items()))
def test_attn_value_head_dim_differs(case):
    B, Hq, Hkv, L, d, dv, kw = case
    (q, k, v, offs, slopes), out, lse = run_attn(B, Hq, Hkv, L, d, seed=L + dv, dv=dv, **kw)
    assert out.shape == (B, Hq, L, dv)
    ro, rl = oracle.attention(q, k, v, **_oracle_kw(kw, offs, slopes))
    check(out, ro, lse, rl)


MULTI_UNIT = [
    # more work units than SMs, so each CTA runs several units back to back
    (2, 16, 16, 1280, 128, dict(mask="causal")),
    (2, 16, 16, 1280, 128, dict()),
    (2, 16, 16, 1280, 32, dict(mask="causal")),
    (2, 16, 16, 1280, 32, dict(score_mod="alibi")),
    (2, 16, 16, 1280, 64, dict(mask="window", window=200)),
]


@pytest.mark.parametrize("case", MULTI_UNIT, ids=lambda c: f"B{c[0]}H{c[1]}L{c[3]}d{c[4]}-" +
                         "-".join(f"{k}{v}" for k, v in c[5].items()))
def test_attn_many_units_per_cta_sampled_rows(case):
    B, Hq, Hkv, L, d, kw = case
    (q, k, v, offs, slopes), out, lse = run_attn(B, Hq, Hkv, L, d, seed=7 + d, **kw)
    rng = np.random.default_rng(d)
    rows = [(int(rng.integers(B)), int(rng.integers(Hq)), int(rng.integers(L))) for _ in range(48)]
    rows += [(0, 0, 0), (B - 1, Hq - 1, L - 1), (1, 3, 127), (1, 5, 128), (0, 9, 1151), (1, 15, 1152)]
    ro, rl = oracle.attention_rows(q, k, v, rows, **_oracle_kw(kw, offs, slopes))
    oc, lc = out.float().cpu(), lse.cpu()
    g = np.stack([oc[b, h, i].numpy() for b, h, i in rows]).astype(np.float64)
    gl = np.array([lc[b, h, i].item() for b, h, i in rows])
    assert np.abs(g - ro).max() <= ATOL and np.linalg.norm(g - ro) / np.linalg.norm(ro) <= RTOL
    assert np.abs(gl - rl).max() <= LSE_ATOL


KEY_SPLIT = [
    # (B, Hq, Hkv, L, d, dv, n_docs, kwargs), run with every unit split along
    # the key axis: the two halves of each query tile's key range are merged
    # through their (m, l) -- odd and even tile counts, single-tile ranges
    # (not split), padding tiles, every mask, both score mods, GQA
    (1, 2, 2, 256, 64, 64, None, dict()),
    (1, 2, 2, 640, 64, 64, None, dict()),
    (2, 3, 3, 300, 64, 64, None, dict(mask="causal")),
    (1, 2, 2, 1000, 64, 64, None, dict(mask="window", window=300)),
    (1, 2, 2, 700, 64, 64, None, dict(mask="prefix_lm", prefix=200)),
    (2, 4, 4, 900, 64, 64, 4, dict(mask="document")),
    (1, 8, 2, 600, 64, 64, None, dict(mask="causal")),
    (1, 6, 2, 520, 64, 64, None, dict()),
    (1, 2, 2, 500, 64, 64, None, dict(score_mod="alibi")),
    (1, 2, 2, 500, 64, 64, None, dict(score_mod="softcap", softcap=20.0)),
    (1, 2, 2, 400, 32, 32, None, dict(mask="causal")),
    (1, 2, 2, 400, 128, 64, None, dict(mask="causal")),
    (1, 2, 2, 300, 64, 32, None, dict()),
]


@pytest.mark.parametrize("case", KEY_SPLIT, ids=lambda c: f"B{c[0]}H{c[1]}x{c[2]}L{c[3]}d{c[4]}dv{c[5]}-" +
                         "-".join(f"{k}{v}" for k, v in c[7].items()))
def test_attn_forced_key_split(case):
    B, Hq, Hkv, L, d, dv, nd, kw = case
    (q, k, v, offs, slopes), out, lse = run_attn(B, Hq, Hkv, L, d, seed=3 * L + d, n_docs=nd, dv=dv,
                                                 debug_flags=FL_DEBUG_KEY_SPLIT, **kw)
    ro, rl = oracle.attention(q, k, v, **_oracle_kw(kw, offs, slopes))
    check(out, ro, lse, rl)


@pytest.mark.parametrize("kw", [dict(), dict(score_mod="softcap", softcap=30.0), dict(mask="window", window=200)],
                         ids=["none", "softcap", "window"])
def test_attn_last_wave_key_split(kw):
    """More units than SMs with a short last wave (at most half the SMs): the
    last wave's units run key-split; the whole output against the oracle."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    # L = 512: two units (query-tile pairs) per head; units = B * H * 2
    H = (sms + 8) // 2
    (q, k, v, offs, slopes), out, lse = run_attn(1, H, H, 512, 64, seed=sms, **kw)
    assert (2 * H) % sms != 0 and 2 * ((2 * H) % sms) <= sms
    ro, rl = oracle.attention(q, k, v, **_oracle_kw(kw, offs, slopes))
    check(out, ro, lse, rl)


def test_causal_row0_is_v0_bit_exact():
    (q, k, v, _, _), out, _ = run_attn(2, 4, 4, 300, 64, seed=5, mask="causal")
    assert torch.equal(out[:, :, 0].cpu(), v[:, :, 0])


def test_identical_keys_give_mean_of_visible_values():
    B, H, L, d = 1, 2, 300, 64
    q, k, v = synth.attn_inputs(B, H, H, L, d, seed=9)
    k = k[:, :, :1].expand(B, H, L, d).contiguous()
    for kw in (dict(), dict(mask="causal"), dict(mask="window", window=50), dict(mask="prefix_lm", prefix=70)):
        out, _ = attn_fwd(*_gpu(q, k, v), **kw)
        vis = oracle.visibility(kw.get("mask", "none"), L, L, window=kw.get("window"), prefix=kw.get("prefix"))
        vv = v.double().numpy()
        ref = np.stack([np.stack([vv[0, h][vis[i]].mean(0) for i in range(L)]) for h in range(H)])[None]
        check(out, ref)


def test_strided_inputs_and_no_lse():
    B, H, L, d = 2, 4, 300, 64
    q, k, v = synth.attn_inputs(B, H, H, L, d, seed=11)
    # [B, L, H, d] storage viewed as [B, H, L, d]
    qs, ks, vs = (t.transpose(1, 2).contiguous().to(DEV).transpose(1, 2) for t in (q, k, v))
    out_store = torch.empty(B, L, H, d, device=DEV, dtype=torch.bfloat16)
    out, lse = attn_fwd(qs, ks, vs, mask="causal", out=out_store.transpose(1, 2), return_lse=False)
    sync_status()
    assert lse is None
    ro, _ = oracle.attention(q, k, v, mask="causal")
    check(out, ro)


def test_repeated_calls_are_deterministic():
    (q, k, v, _, _), out1, lse1 = run_attn(1, 4, 4, 1000, 64, seed=3, mask="causal")
    out2, lse2 = attn_fwd(*_gpu(q, k, v), mask="causal")
    sync_status()
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)


# ----------------------------------------------------------------- diff attn
@pytest.mark.parametrize("B,H,L,causal,lam", [(1, 2, 256, True, 0.8), (2, 3, 300, True, 0.5),
                                               (1, 2, 200, False, 0.8), (1, 1, 1, True, 0.8),
                                               (1, 2, 300, True, 0.0)])
def test_diffattn_small(B, H, L, causal, lam):
    q1, k1, q2, k2, v = synth.diff_inputs(B, H, L, seed=L)
    out, lse = diffattn_fwd(*_gpu(q1, k1, q2, k2, v), lam, causal=causal)
    sync_status()
    ro, r1, r2 = oracle.diff_attention(q1, k1, q2, k2, v, lam, scale=0.125, causal=causal)
    check(out, ro, lse, np.stack([r1, r2]))


# ----------------------------------------------------------------- Evoformer
@pytest.mark.parametrize("B,Ns,Nr,H,d,use_pb,use_mb", [(1, 3, 256, 2, 32, True, True), (2, 2, 100, 3, 32, True, True),
                                                         (1, 2, 300, 2, 32, False, True), (1, 2, 64, 2, 32, True, False),
                                                         (1, 4, 256, 8, 32, True, True), (1, 5, 20, 1, 32, False, False),
                                                         (2, 7, 388, 3, 32, True, True)])
def test_evoformer_small(B, Ns, Nr, H, d, use_pb, use_mb):
    q, k, v, pb, mb, g = synth.evo_inputs(B, Ns, Nr, H, d=d, seed=Nr + d)
    out, lse = evoformer_gated_attn_fwd(*_gpu(q, k, v), pb.to(DEV) if use_pb else None,
                                        mb.to(DEV) if use_mb else None, g.to(DEV))
    sync_status()
    ro, rl = oracle.evoformer_gated_attention(q, k, v, pb if use_pb else np.zeros((B, H, Nr, Nr)),
                                              mb if use_mb else np.zeros((B, Ns, Nr)), g)
    check(out, ro, lse, rl)


@pytest.mark.parametrize("B,Ns,Nr,H,d,use_mb", [(1, 16, 8, 2, 32, True), (1, 128, 12, 3, 32, True),
                                                 (2, 20, 7, 2, 32, True), (1, 200, 6, 2, 32, True),
                                                 (1, 64, 5, 2, 64, True), (1, 33, 4, 2, 32, False),
                                                 (1, 132, 9, 2, 64, False)])
def test_evoformer_col_small(B, Ns, Nr, H, d, use_mb):
    q, k, v, mb, g = synth.evo_col_inputs(B, Ns, Nr, H, d=d, seed=Ns + Nr + d)
    out, lse = evoformer_col_gated_attn_fwd(*_gpu(q, k, v), mb.to(DEV) if use_mb else None, g.to(DEV))
    sync_status()
    ro, rl = oracle.evoformer_col_gated_attention(q, k, v, mb if use_mb else np.zeros((B, Nr, Ns)), g)
    check(out, ro, lse, rl)


# ------------------------------------------------------ bounded-wait failure
def test_skipped_tile_load_times_out_then_recovers():
    q, k, v = synth.attn_inputs(1, 2, 2, 512, 64, seed=1)
    qd, kd, vd = _gpu(q, k, v)
    attn_fwd(qd, kd, vd, debug_flags=FL_DEBUG_SKIP_KV_LOAD, debug_arg=1, wait_limit_ms=20)
    with pytest.raises(FlattnError) as e:
        sync_status()
    assert e.value.status == FL_ERR_TIMEOUT
    out, lse = attn_fwd(qd, kd, vd)
    sync_status()
    ro, rl = oracle.attention(q, k, v)
    check(out, ro, lse, rl)


@pytest.mark.parametrize("L", [1, 17, 129, 255, 300])
def test_output_guard_regions_untouched(L):
    """out and lse placed inside larger buffers whose guard regions hold a
    sentinel; ragged shapes must write exactly their own elements."""
    B, H, d = 1, 2, 64
    q, k, v = synth.attn_inputs(B, H, H, L, d, seed=L)
    pad = 4096  # elements of guard on each side (a multiple of 8: 16-byte aligned)
    n_out, n_lse = B * H * L * d, B * H * L
    obuf = torch.full((pad + n_out + pad,), -7.0, dtype=torch.bfloat16, device=DEV)
    lbuf = torch.full((pad + n_lse + pad,), 12345.0, dtype=torch.float32, device=DEV)
    out = obuf[pad:pad + n_out].view(B, H, L, d)
    lse = lbuf[pad:pad + n_lse].view(B, H, L)
    attn_fwd(*_gpu(q, k, v), mask="causal", out=out, lse=lse)
    sync_status()
    ob, lb = obuf.cpu(), lbuf.cpu()
    assert torch.all(ob[:pad] == -7.0) and torch.all(ob[pad + n_out:] == -7.0)
    assert torch.all(lb[:pad] == 12345.0) and torch.all(lb[pad + n_lse:] == 12345.0)
    ro, rl = oracle.attention(q, k, v, mask="causal")
    check(out, ro, lse, rl)


def test_softcap_both_tanh_paths():
    """Scores inside the polynomial range (|s*scale/cap| <= 0.5) take the FMA
    path, a large-score tile takes the exact MUFU path; both must match."""
    q, k, v = synth.attn_inputs(1, 2, 2, 300, 64, seed=41)
    for cap, qs in ((30.0, 1.0), (2.0, 1.0), (30.0, 40.0)):
        qq = (q.float() * qs).to(torch.bfloat16)
        out, lse = attn_fwd(*_gpu(qq, k, v), score_mod="softcap", softcap=cap)
        sync_status()
        ro, rl = oracle.attention(qq, k, v, score_mod="softcap", softcap=cap)
        check(out, ro, lse, rl)
