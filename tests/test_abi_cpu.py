"""Host-side checks of the C ABI that need no GPU: the library loads, exports every function
declared in include/kda.h, answers size queries, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

from linear_attention_chunked_gb300 import build, kda

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return kda.lib()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "kda.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(kda_\w+)\s*\(", text, flags=re.M)))


def test_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert len(names) >= 7, names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/kda.h but not exported"
    assert set(kda.EXPORTS) <= set(names)


def test_status_strings(lib):
    for s in range(7):
        assert kda.kda_status_string(s)
    assert "unknown" in kda.kda_status_string(99)


def test_workspace_sizes_depend_on_T_N_H_only(lib):
    a = kda.kda_workspace_size(3548, 2, 4, kda.KDA_OP_FWD)
    b = kda.kda_workspace_size(3548, 2, 4, kda.KDA_OP_FWD, gate="raw", l2norm=True)
    assert a == b and a[0] > 0 and a[1] > 0
    fwd, saved = a
    bs, _ = kda.kda_workspace_size(3548, 2, 4, kda.KDA_OP_BWD_SAVED)
    br, _ = kda.kda_workspace_size(3548, 2, 4, kda.KDA_OP_BWD_REPLAY)
    assert fwd <= bs < br and br >= bs + saved
    assert kda.kda_workspace_size(3548, 2, 4, kda.KDA_OP_WALK)[0] == 0
    # grows with T
    assert kda.kda_workspace_size(7096, 2, 4, kda.KDA_OP_FWD)[0] > fwd


@pytest.mark.parametrize("field,value,status", [
    ("H", 0, kda.KDA_ERR_INVALID_ARG),
    ("H", -3, kda.KDA_ERR_INVALID_ARG),
    ("N", 0, kda.KDA_ERR_INVALID_ARG),
    ("T", -1, kda.KDA_ERR_INVALID_ARG),
    ("d", 64, kda.KDA_ERR_UNSUPPORTED),
    ("gate", 7, kda.KDA_ERR_INVALID_ARG),
    ("l2norm", 2, kda.KDA_ERR_INVALID_ARG),
    ("out_fp32", 3, kda.KDA_ERR_INVALID_ARG),
    ("group_chunks", -1, kda.KDA_ERR_INVALID_ARG),
    ("group_chunks", (1 << 20) + 1, kda.KDA_ERR_INVALID_ARG),
])
def test_problem_validation(lib, field, value, status):
    pr = kda.make_problem(128, 1, 2)
    pr.cu_seqlens = 256
    setattr(pr, field, value)
    ws = ctypes.c_size_t(0)
    assert lib.kda_workspace_size(ctypes.byref(pr), 0, ctypes.byref(ws), None) == status
    # the compute entry points validate before any CUDA call
    z = ctypes.c_void_p(0)
    assert lib.kda_fwd(ctypes.byref(pr), *([z] * 11), z, 0, z) == status


def test_pointer_validation(lib):
    pr = kda.make_problem(128, 1, 2)
    pr.cu_seqlens = 256
    z = ctypes.c_void_p(0)
    a = ctypes.c_void_p(4096)
    mis = ctypes.c_void_p(4098)  # not 16-byte aligned
    # null q
    assert lib.kda_fwd(ctypes.byref(pr), z, a, a, a, a, z, z, z, a, z, z, a, 1 << 40, z) == \
        kda.KDA_ERR_INVALID_ARG
    # misaligned k
    assert lib.kda_fwd(ctypes.byref(pr), a, mis, a, a, a, z, z, z, a, z, z, a, 1 << 40, z) == \
        kda.KDA_ERR_INVALID_ARG
    # raw gate needs A_log and dt_bias
    pr.gate = kda.KDA_GATE_RAW
    assert lib.kda_fwd(ctypes.byref(pr), a, a, a, a, a, z, z, z, a, z, z, a, 1 << 40, z) == \
        kda.KDA_ERR_INVALID_ARG
    # workspace too small
    pr.gate = kda.KDA_GATE_G
    assert lib.kda_fwd(ctypes.byref(pr), a, a, a, a, a, z, z, z, a, z, z, a, 16, z) == \
        kda.KDA_ERR_WORKSPACE
    # cu_seqlens null
    pr.cu_seqlens = None
    assert lib.kda_fwd(ctypes.byref(pr), a, a, a, a, a, z, z, z, a, z, z, a, 1 << 40, z) == \
        kda.KDA_ERR_INVALID_ARG
    # walk: N < 1, H < 1, bad reverse flag, unknown product format, misaligned status pointer
    assert lib.kda_transfer_walk(0, a, 1, 1, a, a, z, 0, 0, a, z, z, z) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_transfer_walk(1, a, 1, 0, a, a, z, 0, 0, a, z, z, z) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_transfer_walk(1, a, 1, 1, a, a, z, 2, 0, a, z, z, z) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_transfer_walk(1, a, 1, 1, a, a, z, 0, 5, a, z, z, z) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_transfer_walk(1, a, 1, 1, a, a, z, 0, -1, a, z, z, z) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_transfer_walk(1, a, 1, 1, a, a, z, 0, 0, a, z, ctypes.c_void_p(258), z) == \
        kda.KDA_ERR_INVALID_ARG
    # fragment summary: bad mode
    pf = kda.make_problem(128, 1, 2)
    pf.cu_seqlens = 256
    assert lib.kda_fragment_summary(ctypes.byref(pf), 5, *([a] * 10), a, 1 << 40, z) == \
        kda.KDA_ERR_INVALID_ARG


def test_output_dtype_must_match_the_declared_one():
    import torch
    kda._check_dtypes({"o": torch.empty(2, dtype=torch.bfloat16)}, torch.bfloat16)
    with pytest.raises(ValueError, match="dq is torch.float32"):
        kda._check_dtypes({"dq": torch.empty(2, dtype=torch.float32)}, torch.bfloat16)


def test_selftest_wait_timeout_validation(lib):
    # argument checks come before any CUDA call (a null workspace, a limit out of range)
    assert lib.kda_selftest_wait_timeout(None, ctypes.c_uint32(1000), None) == kda.KDA_ERR_INVALID_ARG
    buf = (ctypes.c_char * 64)()
    aligned = ctypes.addressof(buf) + (-ctypes.addressof(buf)) % 16
    assert lib.kda_selftest_wait_timeout(ctypes.c_void_p(aligned), ctypes.c_uint32(0), None) == \
        kda.KDA_ERR_INVALID_ARG
    assert lib.kda_selftest_wait_timeout(ctypes.c_void_p(aligned), ctypes.c_uint32(2000000), None) == \
        kda.KDA_ERR_INVALID_ARG


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    # no fallback of any kind: without the built library every entry point raises
    from linear_attention_chunked_gb300 import build, kda
    monkeypatch.setattr(kda, "_lib", None)
    monkeypatch.setattr(build, "LIB", str(tmp_path / "libkda_gb300.so"))
    with pytest.raises(RuntimeError, match="is missing"):
        kda.lib()
    with pytest.raises(RuntimeError, match="is missing"):
        kda.kda_status_string(0)


def test_chunk_group_sizes_and_entry_points(lib):
    # the group region grows every op's workspace and the saved set (the groups' M); sizes still
    # depend on (T, N, H, group_chunks) only
    base = {op: kda.kda_workspace_size(16384, 4, 64, op) for op in
            (kda.KDA_OP_FWD, kda.KDA_OP_BWD_SAVED, kda.KDA_OP_BWD_REPLAY)}
    grp = {op: kda.kda_workspace_size(16384, 4, 64, op, group_chunks=48) for op in base}
    for op in base:
        assert grp[op][0] > base[op][0] and grp[op][1] > base[op][1]
    # Gmax = N + ceil((ceil(T / 64) + N) / G) = 4 + ceil(260 / 48) = 10 groups: three
    # [Gmax][H][128][128] fp32 arrays in the workspace, one in the saved set
    g_state = 10 * 64 * 128 * 128 * 4
    assert 3 * g_state <= grp[kda.KDA_OP_FWD][0] - base[kda.KDA_OP_FWD][0] < 3 * g_state + 4096
    assert g_state <= grp[kda.KDA_OP_FWD][1] - base[kda.KDA_OP_FWD][1] < g_state + 512
    # the fragment summaries and the allocation-free forward take group_chunks = 0 only
    pr = kda.make_problem(128, 1, 2, group_chunks=2)
    pr.cu_seqlens = 256
    z = ctypes.c_void_p(0)
    assert lib.kda_fragment_summary(ctypes.byref(pr), 0, *([z] * 10), z, 0, z) == kda.KDA_ERR_UNSUPPORTED
    assert lib.kda_fwd_static_ws(ctypes.byref(pr), *([z] * 10), z) == kda.KDA_ERR_UNSUPPORTED


def test_conv_validation(lib):
    ws = ctypes.c_size_t(0)
    pr = kda.make_conv_problem(1000, 2, 64)
    pr.cu_seqlens = 256
    assert lib.kda_conv_workspace_size(ctypes.byref(pr), ctypes.byref(ws)) == kda.KDA_OK
    # partial sums of dw (4) and dbias (1) per channel for every 512-token block row
    assert ws.value >= 2 * 5 * 64 * 4
    for field, value in (("C", 12), ("C", 0), ("N", 0), ("T", -1), ("T", (1 << 31) - 1),
                         ("activation", 2), ("out_fp32", 5)):
        bad = kda.make_conv_problem(1000, 2, 64)
        bad.cu_seqlens = 256
        setattr(bad, field, value)
        assert lib.kda_conv_workspace_size(ctypes.byref(bad), ctypes.byref(ws)) == \
            kda.KDA_ERR_INVALID_ARG, (field, value)
    z = ctypes.c_void_p(0)
    a = ctypes.c_void_p(4096)
    mis = ctypes.c_void_p(4104)
    # null x / y, misaligned w, a halo gradient without a halo, workspace too small
    assert lib.kda_conv_fwd(ctypes.byref(pr), z, a, z, z, a, z) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_conv_fwd(ctypes.byref(pr), a, a, z, z, z, z) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_conv_fwd(ctypes.byref(pr), a, mis, z, z, a, z) == kda.KDA_ERR_INVALID_ARG
    assert lib.kda_conv_bwd(ctypes.byref(pr), a, a, z, z, a, a, a, z, a, a, 1 << 30, z) == \
        kda.KDA_ERR_INVALID_ARG
    assert lib.kda_conv_bwd(ctypes.byref(pr), a, a, z, z, a, a, a, z, z, a, 16, z) == \
        kda.KDA_ERR_WORKSPACE
