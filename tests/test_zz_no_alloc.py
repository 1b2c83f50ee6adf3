"""The allocation-free forward, kda_fwd_static_ws, against the regular kda_fwd.

kda_fwd_static_ws is for callers that cannot allocate device memory (the library's own static
device array is its scratch, so the caller passes only inputs and outputs).  Two calls in a row,
on different problems, must match kda_fwd within the parity tolerances the other tests use; a
problem larger than the static scratch must be refused before anything runs.  This file is
collected last so that a run stopping at the first failure has run every other test already."""
import numpy as np
import pytest
import torch

from harness import TOL, rel_err, to_dev
from linear_attention_chunked_gb300 import inputs, kda

pytestmark = pytest.mark.gpu


def _run_both(inp, gate, l2n):
    d = to_dev(inp)
    a = (d["q"], d["k"], d["v"], d["beta"], d["g"], d["cu_seqlens"])
    kw = dict(gate=gate, A_log=d["A_log"], dt_bias=d["dt_bias"], l2norm=l2n)
    o_s, ht_s = kda.kda_fwd_static_ws(*a, **kw)
    o_r, ht_r, _ = kda.kda_fwd(*a, **kw, save=False)
    torch.cuda.synchronize()
    return [x.float().cpu().numpy() for x in (o_s, ht_s, o_r, ht_r)]


def test_static_ws_forward_matches_kda_fwd_two_calls():
    cases = [
        (inputs.make_inputs([130, 1, 65], 2, gate="raw", l2norm=True, seed=21), "raw", True),
        (inputs.make_inputs([200, 77], 3, gate="g", l2norm=False, seed=22), "g", False),
    ]
    for inp, gate, l2n in cases:
        o_s, ht_s, o_r, ht_r = _run_both(inp, gate, l2n)
        assert np.isfinite(o_s).all() and np.isfinite(ht_s).all()
        assert rel_err(o_s, o_r) <= TOL["o"], rel_err(o_s, o_r)
        assert rel_err(ht_s, ht_r) <= TOL["ht"], rel_err(ht_s, ht_r)


def test_static_ws_rejects_too_large():
    T, N, H = 16384, 1, 64  # needs far more than the static scratch
    ws, _ = kda.kda_workspace_size(T, N, H, kda.KDA_OP_FWD)
    assert ws > kda.KDA_STATIC_WS_BYTES
    q = torch.zeros((T, H, 128), dtype=torch.bfloat16, device="cuda")
    g = torch.zeros((T, H, 128), dtype=torch.float32, device="cuda")
    beta = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    cu = torch.tensor([0, T], dtype=torch.int32, device="cuda")
    with pytest.raises(kda.KdaError) as e:
        kda.kda_fwd_static_ws(q, q, q, beta, g, cu)
    assert e.value.status == kda.KDA_ERR_TOO_LARGE
