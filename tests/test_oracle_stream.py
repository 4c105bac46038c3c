"""Streaming FS-L decoding from a bounded state (oracle.stream) against the
definition-form forward over the whole history (CPU).

The pages describe FS-L's pool as bounded (at most 72 cells) and updated only
at query-block boundaries, with a bounded state and a streaming cache that
stays constant with context length ("FreeSolo: Linear-time Sparse Attention
with Zero-Shot Length Extrapolation": ai.info summary, "Methodology in Plain
English"; paper.rainbus.top summary, 核心方法 and 实验结果).  Decoding token by
token while holding only the window, the open and pending cells, the recent
cells and the running top-P cells must reproduce every row of the full
forward (same selections, outputs to float64 rounding), and the rows held
must stay under a bound that does not grow with N."""
import numpy as np
import pytest

from oracle import oracle
from oracle.stream import decode_stream

TINY = dict(w=24, s=8, K=2, P=4, W=2, Bq=32, rope_base=10000.0, rms_eps=1e-6, mode=0)
PAGE = dict(oracle.DEFAULT_PARAMS)


@pytest.mark.parametrize("params,N,d,seed", [(TINY, 512, 8, 1), (TINY, 1024, 8, 2),
                                             (PAGE, 2048, 64, 3)])
def test_stream_decode_matches_full_forward(params, N, d, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((1, N, d)).astype(np.float32)
    k = (rng.standard_normal((1, N, d)) * np.exp(0.5 * rng.standard_normal((1, N, 1))))
    k = k.astype(np.float32)
    v = rng.standard_normal((1, N, d)).astype(np.float32)
    lam, sig, mix = 0.9, 4.0, 0.6
    ref = oracle.forward(q, k, v, 1, [lam], [sig], [mix], params=params, want_branches=False)
    out, sel, held, bound = decode_stream(q[0], k[0], v[0], lam, sig, mix, params)
    ties = ref["gap_rel"][0] < 1e-12
    assert np.array_equal(sel[~ties], ref["sel"][0][~ties])
    np.testing.assert_allclose(out[~ties], ref["out"][0][~ties], rtol=1e-11, atol=1e-12)
    assert held <= bound


def test_stream_state_does_not_grow_with_length():
    rng = np.random.default_rng(7)
    held = []
    for N in (1024, 2048):
        q = rng.standard_normal((N, 8)).astype(np.float32)
        k = rng.standard_normal((N, 8)).astype(np.float32)
        v = rng.standard_normal((N, 8)).astype(np.float32)
        _, _, h, bound = decode_stream(q, k, v, 1.0, 4.0, 0.5, TINY)
        held.append(h)
    assert held[0] == held[1] <= bound  # reached at the first full pool, then flat
