"""The allocation-free forward, kda_fwd_static_ws, against the regular kda_fwd.

kda_fwd_static_ws serves callers that cannot allocate device memory: code running inside a host
runtime that owns every device allocation and hands an op no workspace, or code that must not
grow the footprint behind the caller's allocator.  Its scratch is the library's own static
device array, so the caller passes only inputs and outputs.  It runs the same kernels as kda_fwd
without a saved set, on the same inputs, so its outputs must be bitwise equal to kda_fwd's --
also on the second of two calls in a row on different problems, where a dependence on what the
previous call left in the shared array would show.  A call allocates nothing: the device's free
memory is the same before and after it.  A problem larger than the static scratch is refused
before anything runs.  This file is collected last, so a run that stops at the first failure
has run every other test already; it also passes alone in a fresh process."""
import numpy as np
import pytest
import torch

from harness import to_dev
from linear_attention_chunked_gb300 import inputs, kda

pytestmark = pytest.mark.gpu


def _args(inp, gate, l2n):
    d = to_dev(inp)
    a = (d["q"], d["k"], d["v"], d["beta"], d["g"], d["cu_seqlens"])
    kw = dict(gate=gate, A_log=d["A_log"], dt_bias=d["dt_bias"], l2norm=l2n)
    return a, kw


def test_static_ws_forward_bitwise_equals_kda_fwd_two_calls():
    cases = [
        (inputs.make_inputs([130, 1, 65], 2, gate="raw", l2norm=True, seed=21), "raw", True),
        (inputs.make_inputs([200, 77], 3, gate="g", l2norm=False, seed=22), "g", False),
    ]
    for inp, gate, l2n in cases:  # two calls in a row, each followed by the regular forward
        a, kw = _args(inp, gate, l2n)
        o_s, ht_s = kda.kda_fwd_static_ws(*a, **kw)
        o_r, ht_r, _ = kda.kda_fwd(*a, **kw, save=False)
        torch.cuda.synchronize()
        o_s, ht_s, o_r, ht_r = (x.cpu().numpy() for x in (o_s, ht_s, o_r, ht_r))
        assert np.isfinite(o_s).all() and np.isfinite(ht_s).all()
        assert np.array_equal(o_s, o_r)
        assert np.array_equal(ht_s, ht_r)


def test_static_ws_call_allocates_no_device_memory():
    inp = inputs.make_inputs([190, 66], 2, gate="raw", l2norm=False, seed=23)
    a, kw = _args(inp, "raw", False)
    o = torch.empty(a[0].shape, dtype=torch.float32, device="cuda")
    ht = torch.empty((2, 2, 128, 128), dtype=torch.float32, device="cuda")
    kda.kda_fwd_static_ws(*a, **kw, o=o, ht=ht)  # first call: device set-up, code loaded
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    kda.kda_fwd_static_ws(*a, **kw, o=o, ht=ht)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    o_r, ht_r, _ = kda.kda_fwd(*a, **kw, save=False)
    torch.cuda.synchronize()
    assert torch.equal(o, o_r) and torch.equal(ht, ht_r)


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
