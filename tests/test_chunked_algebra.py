"""The chunk-parallel algebra used by the CUDA kernels, written in float64 numpy
(tests/chunked_ref.py), equals the token-by-token oracle.  This separates "is the decomposition
right" from "is the kernel right": a GPU mismatch with this test green is a kernel bug."""
import numpy as np
import pytest

import oracle
from chunked_ref import kda_chunked


@pytest.mark.parametrize("raw,l2n,chunk,lens", [
    (False, False, 64, [130, 5, 64]),
    (True, False, 16, [40, 1, 17]),
    (False, True, 16, [33, 16]),
    (True, True, 8, [19, 0, 9]),
])
def test_chunked_equals_oracle(raw, l2n, chunk, lens):
    rng = np.random.default_rng(30)
    H, d = 2, 16
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    q = rng.standard_normal((T, H, d))
    k = rng.standard_normal((T, H, d))
    if not l2n:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, d))
    beta = 1 / (1 + np.exp(-rng.standard_normal((T, H))))
    if raw:
        g = rng.standard_normal((T, H, d))
        A_log = rng.uniform(0, np.log(16), H)
        dt_bias = rng.uniform(-1, 1, (H, d))
    else:
        g = -0.1 * np.abs(rng.standard_normal((T, H, d)))
        A_log = dt_bias = None
    h0 = rng.standard_normal((len(lens), H, d, d))
    dht = rng.standard_normal((len(lens), H, d, d))
    dO = rng.standard_normal((T, H, d))
    kw = dict(raw=raw, A_log=A_log, dt_bias=dt_bias, h0=h0, l2norm=l2n)
    o, ht, gr = kda_chunked(q, k, v, beta, g, cu, dO, dht=dht, chunk=chunk, **kw)
    o_ref, ht_ref = oracle.kda_fwd(q, k, v, beta, g, cu, **kw)
    g_ref = oracle.kda_bwd(q, k, v, beta, g, cu, dO, dht=dht, **kw)
    np.testing.assert_allclose(o, o_ref, rtol=1e-9, atol=1e-10)
    np.testing.assert_allclose(ht, ht_ref, rtol=1e-9, atol=1e-10)
    for name, ref in g_ref.items():
        err = np.max(np.abs(gr[name] - ref)) / max(np.max(np.abs(ref)), 1e-30)
        assert err < 1e-9, f"{name}: {err:.3e}"
