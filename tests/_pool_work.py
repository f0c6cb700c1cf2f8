"""Worker functions for the oracle process pool of the whole-tensor parity
tests (imported by spawned workers; test infrastructure only)."""
import os

os.environ.setdefault("OMP_NUM_THREADS", "1")
os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")


def attention_head(args):
    """oracle.attention on one (batch, head) slice: args = (q, k, v, kw)
    with numpy arrays [1, 1, L, d]; returns (out [L, dv], lse [L])."""
    import oracle
    q, k, v, kw = args
    o, l = oracle.attention(q, k, v, **kw)
    return o[0, 0], l[0, 0]
