"""GPU parity of the decode-phase (key/value cache) attention against the
fp64 oracle, through the C ABI: every output element and LSE compared with
the same bar as the other parity tests (max-abs <= 2e-2, relative L2 <=
1e-2, LSE max-abs <= 1e-3)."""
import numpy as np
import pytest
import torch

import oracle
from flashattention_attn_fwd_gb300 import attn_decode_fwd, synth, sync_status

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _check(out, lse, ro, rl):
    g = out.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(g).all()
    err = np.abs(g - ro)
    norm = np.linalg.norm(ro)
    assert err.max() <= 2e-2, err.max()
    if norm > 0:
        assert np.linalg.norm(g - ro) / norm <= 1e-2
    gl = lse.cpu().numpy().astype(np.float64)
    fin = np.isfinite(rl)
    assert (np.isfinite(gl) == fin).all()
    if fin.any():
        assert np.abs(gl[fin] - rl[fin]).max() <= 1e-3


CASES = [
    # (B, Hq, Hkv, Lq, Lmax, d, kwargs)
    (2, 8, 2, 1, 300, 64, dict()),
    (2, 8, 2, 1, 300, 64, dict(causal=True)),
    (3, 4, 4, 1, 1000, 128, dict()),
    (2, 32, 8, 1, 2048, 64, dict()),
    (2, 8, 2, 4, 700, 64, dict(causal=True)),
    (1, 16, 2, 4, 513, 128, dict(causal=True)),
    (2, 8, 2, 2, 900, 64, dict(causal=True, score_mod="alibi")),
    (2, 8, 2, 1, 640, 64, dict(score_mod="softcap", softcap=5.0)),
    (4, 4, 1, 16, 256, 64, dict(causal=True)),
    (1, 64, 1, 1, 129, 64, dict()),
    (2, 8, 2, 1, 100, 64, dict(causal=True)),
    (2, 16, 2, 1, 1500, 128, dict(score_mod="alibi")),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"B{c[0]}H{c[1]}x{c[2]}Lq{c[3]}L{c[4]}d{c[5]}-" +
                         "-".join(f"{k}{v}" for k, v in c[6].items()))
def test_decode_small(case):
    B, Hq, Hkv, Lq, Lmax, d, kw = case
    q, k, v, kv_len = synth.decode_inputs(B, Hq, Hkv, Lq, Lmax, d, seed=Lmax + d + Lq)
    gkw = dict(kw)
    okw = dict(kw)
    if kw.get("score_mod") == "alibi":
        s = synth.alibi_slopes(Hq)
        gkw["alibi_slopes"], okw["slopes"] = s.to(DEV), s
    out, lse = attn_decode_fwd(q.to(DEV), k.to(DEV), v.to(DEV), kv_len.to(DEV), **gkw)
    sync_status()
    ro, rl = oracle.decode_attention(q, k, v, kv_len, **okw)
    _check(out, lse, ro, rl)


def test_decode_edge_lengths_and_full_cache():
    """kv_len of 0 (no visible key: out 0, lse -inf), 1, exactly the
    capacity, and no kv_len array at all."""
    B, Hq, Hkv, Lq, Lmax, d = 4, 8, 2, 1, 384, 64
    q, k, v, _ = synth.decode_inputs(B, Hq, Hkv, Lq, Lmax, d, seed=5)
    kv_len = torch.tensor([0, 1, 384, 200], dtype=torch.int32)
    out, lse = attn_decode_fwd(q.to(DEV), k.to(DEV), v.to(DEV), kv_len.to(DEV))
    sync_status()
    ro, rl = oracle.decode_attention(q, k, v, kv_len)
    _check(out, lse, ro, rl)
    assert torch.all(out[0].cpu() == 0) and torch.all(torch.isinf(lse[0].cpu()))
    out2, lse2 = attn_decode_fwd(q.to(DEV), k.to(DEV), v.to(DEV), None)
    sync_status()
    ro2, rl2 = oracle.decode_attention(q, k, v, None)
    _check(out2, lse2, ro2, rl2)


def test_decode_serving_batch_whole_tensor():
    """The LLaMA-3.2-1B-shaped decode batch the benchmark times (B=16,
    Hq=32, Hkv=8, d=64, cache capacity 8192, mixed lengths), every element."""
    B, Hq, Hkv, Lq, Lmax, d = 16, 32, 8, 1, 8192, 64
    q, k, v, kv_len = synth.decode_inputs(B, Hq, Hkv, Lq, Lmax, d, seed=61)
    out, lse = attn_decode_fwd(q.to(DEV), k.to(DEV), v.to(DEV), kv_len.to(DEV))
    sync_status()
    ro, rl = oracle.decode_attention(q, k, v, kv_len)
    _check(out, lse, ro, rl)


def test_decode_workspace_matches_the_split_rule():
    """fl_attn_decode_workspace_size against the split rule on this GPU's SM
    count: four CTAs per SM with up to 8 query rows per CTA, sixteen with
    more; fp32 partial output and log-sum-exp per split and row."""
    import ctypes
    from flashattention_attn_fwd_gb300 import _lib
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for B, Hq, Hkv, Lq, Lmax, d in ((16, 32, 8, 1, 8192, 64), (4, 32, 2, 1, 4096, 128), (2, 8, 2, 8, 2048, 64),
                                    (1, 4, 4, 1, 100, 64)):
        M = Hq // Hkv * Lq
        tiles = (Lmax + 127) // 128
        ns = max(1, min(tiles, -(-(4 if M <= 8 else 16) * sms // (B * Hkv))))
        per = -(-tiles // ns)
        ns = -(-tiles // per)
        want = 0 if ns <= 1 else ns * B * Hq * Lq * (d + 1) * 4
        desc = _lib.new_desc()
        desc.B, desc.Hq, desc.Hkv, desc.Lq, desc.Lk, desc.d, desc.dv = B, Hq, Hkv, Lq, Lmax, d, d
        assert _lib.lib().fl_attn_decode_workspace_size(ctypes.byref(desc)) == want
