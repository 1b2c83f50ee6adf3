"""ctypes binding of the C ABI in include/kda.h (argument marshalling only).

Every function here has the name of the C entry point it calls.  PyTorch supplies device memory
and the current stream; all arithmetic runs in the CUDA kernels of libkda_gb300.so.  If that
library has not been built this module raises -- there is no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

D = 128
CHUNK = 64

KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, KDA_ERR_WORKSPACE = 0, 1, 2, 3
KDA_ERR_CUDA, KDA_ERR_TIMEOUT, KDA_ERR_DEVICE_CHECK, KDA_ERR_TOO_LARGE = 4, 5, 6, 7
KDA_STATIC_WS_BYTES = 64 << 20
KDA_GATE_G, KDA_GATE_RAW = 0, 1
KDA_OP_FWD, KDA_OP_BWD_SAVED, KDA_OP_BWD_REPLAY, KDA_OP_FRAGMENT, KDA_OP_WALK = 0, 1, 2, 3, 4
KDA_FRAG_FWD, KDA_FRAG_BWD = 0, 1
KDA_WALK_FP32, KDA_WALK_TF32, KDA_WALK_TF32_HILO, KDA_WALK_BF16X3, KDA_WALK_BF16X3_HW = 0, 1, 2, 3, 4
WALK_PRECISIONS = {"fp32": KDA_WALK_FP32, "tf32": KDA_WALK_TF32, "tf32_hilo": KDA_WALK_TF32_HILO,
                   "bf16x3": KDA_WALK_BF16X3, "bf16x3_hw": KDA_WALK_BF16X3_HW}
WALK_DEFAULT = KDA_WALK_BF16X3_HW  # the format the pages ship as the default walk

EXPORTS = ("kda_workspace_size", "kda_fwd", "kda_fwd_static_ws", "kda_bwd", "kda_fragment_summary",
           "kda_transfer_walk", "kda_conv_workspace_size", "kda_conv_fwd", "kda_conv_bwd",
           "kda_read_device_status", "kda_profile_enable",
           "kda_profile_collect", "kda_kernel_count", "kda_kernel_name", "kda_launch_counter",
           "kda_status_string")


class KdaError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn}: {kda_status_string(status)} (status {status})")


class kda_conv_problem(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("N", ctypes.c_int32), ("C", ctypes.c_int32),
                ("activation", ctypes.c_int32), ("out_fp32", ctypes.c_int32),
                ("cu_seqlens", ctypes.c_void_p)]


class kda_problem(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("N", ctypes.c_int32), ("H", ctypes.c_int32),
                ("d", ctypes.c_int32), ("gate", ctypes.c_int32), ("l2norm", ctypes.c_int32),
                ("out_fp32", ctypes.c_int32), ("group_chunks", ctypes.c_int32),
                ("scale", ctypes.c_float), ("l2_eps", ctypes.c_float),
                ("cu_seqlens", ctypes.c_void_p)]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def lib():
    """Loads libkda_gb300.so (raises if it was not built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if not os.path.exists(path):
                raise RuntimeError(f"CUDA library {path} is missing: run "
                                   "`python -m linear_attention_chunked_gb300.build` first")
            L = ctypes.CDLL(path)
            P, I, S, V = ctypes.POINTER(kda_problem), ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p
            L.kda_workspace_size.argtypes = [P, I, ctypes.POINTER(S), ctypes.POINTER(S)]
            L.kda_fwd.argtypes = [P] + [V] * 11 + [V, S, V]
            L.kda_fwd_static_ws.argtypes = [P] + [V] * 10 + [V]
            L.kda_bwd.argtypes = [P] + [V] * 19 + [V, S, V]
            L.kda_fragment_summary.argtypes = [P, I] + [V] * 10 + [V, S, V]
            L.kda_transfer_walk.argtypes = [ctypes.c_int32, V, ctypes.c_int32, ctypes.c_int32,
                                            V, V, V, I, I, V, V, V, V]
            CP = ctypes.POINTER(kda_conv_problem)
            L.kda_conv_workspace_size.argtypes = [CP, ctypes.POINTER(S)]
            L.kda_conv_fwd.argtypes = [CP, V, V, V, V, V, V]
            L.kda_conv_bwd.argtypes = [CP] + [V] * 9 + [V, S, V]
            L.kda_read_device_status.argtypes = [V, ctypes.POINTER(I), V]
            L.kda_selftest_wait_timeout.argtypes = [V, ctypes.c_uint32, V]
            L.kda_profile_enable.argtypes = [I]
            L.kda_profile_collect.argtypes = [V, V]
            L.kda_kernel_count.argtypes = []
            L.kda_kernel_name.argtypes = [I]
            L.kda_kernel_name.restype = ctypes.c_char_p
            L.kda_launch_counter.argtypes = []
            L.kda_launch_counter.restype = ctypes.c_uint64
            L.kda_status_string.argtypes = [I]
            L.kda_status_string.restype = ctypes.c_char_p
            for name in ("kda_workspace_size", "kda_fwd", "kda_fwd_static_ws", "kda_bwd", "kda_fragment_summary",
                         "kda_transfer_walk", "kda_conv_workspace_size", "kda_conv_fwd",
                         "kda_conv_bwd", "kda_read_device_status", "kda_selftest_wait_timeout",
                         "kda_profile_enable",
                         "kda_profile_collect", "kda_kernel_count"):
                getattr(L, name).restype = ctypes.c_int
            _lib = L
    return _lib


def kda_status_string(status: int) -> str:
    return lib().kda_status_string(int(status)).decode()


def _check(fn, status):
    if status != KDA_OK:
        raise KdaError(fn, status)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _gate(gate):
    if gate in ("g", KDA_GATE_G):
        return KDA_GATE_G
    if gate in ("raw", KDA_GATE_RAW):
        return KDA_GATE_RAW
    raise ValueError(f"gate must be 'g' or 'raw', got {gate!r}")


def make_problem(T, N, H, cu_seqlens=None, *, gate="g", l2norm=False, scale=1.0, eps=1e-6,
                 d=D, out_dtype=torch.float32, group_chunks=0):
    if out_dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("out_dtype must be torch.float32 or torch.bfloat16")
    return kda_problem(int(T), int(N), int(H), int(d), _gate(gate), int(bool(l2norm)),
                       int(out_dtype == torch.float32), int(group_chunks), float(scale), float(eps),
                       None if cu_seqlens is None else cu_seqlens.data_ptr())


def kda_workspace_size(T, N, H, op, **kw):
    """Returns (workspace bytes, saved-set bytes) of op for (T, N, H)."""
    pr = make_problem(T, N, H, **kw)
    if pr.cu_seqlens is None:
        pr.cu_seqlens = 16  # size queries never read it; any aligned non-null value passes
    ws, sv = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check("kda_workspace_size",
           lib().kda_workspace_size(ctypes.byref(pr), int(op), ctypes.byref(ws), ctypes.byref(sv)))
    return ws.value, sv.value


def _check_dtypes(tensors, dtype):
    """The library writes outputs in the dtype the problem declares: a caller's tensor must match."""
    for name, t in tensors.items():
        if t.dtype != dtype:
            raise ValueError(f"{name} is {t.dtype}, the call writes {dtype}")


def _empty_bytes(n, device):
    return torch.empty(max(int(n), 256), dtype=torch.uint8, device=device)


def _shape(q, cu_seqlens):
    T, H, d = q.shape
    return T, cu_seqlens.numel() - 1, H, d


def kda_fwd(q, k, v, beta, g_or_a, cu_seqlens, *, gate="g", A_log=None, dt_bias=None, h0=None,
            l2norm=False, scale=1.0, eps=1e-6, save=True, out_dtype=torch.float32, o=None, ht=None,
            saved=None, ws=None, group_chunks=0):
    """Forward.  Returns (o, ht, saved) -- saved is None when save=False.  group_chunks > 0 cuts
    documents into groups of that many chunks whose summaries are composed by the walk."""
    T, N, H, d = _shape(q, cu_seqlens)
    dev = q.device
    pr = make_problem(T, N, H, cu_seqlens, gate=gate, l2norm=l2norm, scale=scale, eps=eps, d=d,
                      out_dtype=out_dtype, group_chunks=group_chunks)
    ws_b, sv_b = kda_workspace_size(T, N, H, KDA_OP_FWD, group_chunks=group_chunks)
    if ws is None:
        ws = _empty_bytes(ws_b, dev)
    if save and saved is None:
        saved = _empty_bytes(sv_b, dev)
    if not save:
        saved = None
    if o is None:
        o = torch.empty(q.shape, dtype=out_dtype, device=dev)
    _check_dtypes({"o": o}, out_dtype)
    if ht is None:
        ht = torch.empty((N, H, d, d), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        st = lib().kda_fwd(ctypes.byref(pr), _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g_or_a),
                           _ptr(A_log), _ptr(dt_bias), _ptr(h0), _ptr(o), _ptr(ht), _ptr(saved),
                           _ptr(ws), ws.numel(), _stream(dev))
    _check("kda_fwd", st)
    return o, ht, saved


def kda_fwd_static_ws(q, k, v, beta, g_or_a, cu_seqlens, *, gate="g", A_log=None, dt_bias=None,
                      h0=None, l2norm=False, scale=1.0, eps=1e-6, out_dtype=torch.float32,
                      o=None, ht=None):
    """Forward through the allocation-free entry point (its scratch is a static device array of
    the library).  Returns (o, ht).  The output tensors are the caller's (allocated here when not
    given, as any caller would); the library itself allocates nothing."""
    T, N, H, d = _shape(q, cu_seqlens)
    dev = q.device
    pr = make_problem(T, N, H, cu_seqlens, gate=gate, l2norm=l2norm, scale=scale, eps=eps, d=d,
                      out_dtype=out_dtype)
    if o is None:
        o = torch.empty(q.shape, dtype=out_dtype, device=dev)
    _check_dtypes({"o": o}, out_dtype)
    if ht is None:
        ht = torch.empty((N, H, d, d), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        st = lib().kda_fwd_static_ws(ctypes.byref(pr), _ptr(q), _ptr(k), _ptr(v), _ptr(beta),
                                     _ptr(g_or_a), _ptr(A_log), _ptr(dt_bias), _ptr(h0), _ptr(o),
                                     _ptr(ht), _stream(dev))
    _check("kda_fwd_static_ws", st)
    return o, ht


def kda_bwd(q, k, v, beta, g_or_a, cu_seqlens, dO, *, saved=None, gate="g", A_log=None,
            dt_bias=None, h0=None, dht=None, l2norm=False, scale=1.0, eps=1e-6, want_dh0=True,
            out_dtype=torch.float32, out=None, ws=None, group_chunks=0):
    """Backward (saved=None: checkpoint replay).  Returns a dict of gradients.  group_chunks must
    be the forward's."""
    T, N, H, d = _shape(q, cu_seqlens)
    dev = q.device
    g_ = _gate(gate)
    pr = make_problem(T, N, H, cu_seqlens, gate=gate, l2norm=l2norm, scale=scale, eps=eps, d=d,
                      out_dtype=out_dtype, group_chunks=group_chunks)
    op = KDA_OP_BWD_SAVED if saved is not None else KDA_OP_BWD_REPLAY
    ws_b, _ = kda_workspace_size(T, N, H, op, group_chunks=group_chunks)
    if ws is None:
        ws = _empty_bytes(ws_b, dev)
    if out is None:
        od = dict(dtype=out_dtype, device=dev)
        out = dict(dq=torch.empty(q.shape, **od), dk=torch.empty(k.shape, **od),
                   dv=torch.empty(v.shape, **od), dbeta=torch.empty(beta.shape, **od),
                   dg=torch.empty_like(g_or_a))
        if g_ == KDA_GATE_RAW:
            out["dA_log"] = torch.empty((H,), dtype=torch.float32, device=dev)
            out["ddt_bias"] = torch.empty((H, d), dtype=torch.float32, device=dev)
        if want_dh0:
            out["dh0"] = torch.empty((N, H, d, d), dtype=torch.float32, device=dev)
    _check_dtypes({k: out[k] for k in ("dq", "dk", "dv", "dbeta")}, out_dtype)
    _check_dtypes({k: out[k] for k in ("dg", "dA_log", "ddt_bias", "dh0") if out.get(k) is not None},
                  torch.float32)
    with torch.cuda.device(dev):
        st = lib().kda_bwd(ctypes.byref(pr), _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g_or_a),
                           _ptr(A_log), _ptr(dt_bias), _ptr(h0), _ptr(dO), _ptr(dht), _ptr(saved),
                           _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]), _ptr(out["dbeta"]),
                           _ptr(out["dg"]), _ptr(out.get("dA_log")), _ptr(out.get("ddt_bias")),
                           _ptr(out.get("dh0")), _ptr(ws), ws.numel(), _stream(dev))
    _check("kda_bwd", st)
    return out


def kda_fragment_summary(q, k, v, beta, g_or_a, frag_cu, *, mode=KDA_FRAG_FWD, dO=None,
                         gate="g", A_log=None, dt_bias=None, l2norm=False, scale=1.0, eps=1e-6,
                         M=None, B_or_C=None, ws=None):
    """mode KDA_FRAG_FWD -> (M, B); mode KDA_FRAG_BWD -> C.  Fragments = documents of frag_cu."""
    T, F, H, d = _shape(q, frag_cu)
    dev = q.device
    pr = make_problem(T, F, H, frag_cu, gate=gate, l2norm=l2norm, scale=scale, eps=eps, d=d)
    ws_b, _ = kda_workspace_size(T, F, H, KDA_OP_FRAGMENT)
    if ws is None:
        ws = _empty_bytes(ws_b, dev)
    if mode == KDA_FRAG_FWD and M is None:
        M = torch.empty((F, H, d, d), dtype=torch.float32, device=dev)
    if B_or_C is None:
        B_or_C = torch.empty((F, H, d, d), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        st = lib().kda_fragment_summary(ctypes.byref(pr), int(mode), _ptr(q), _ptr(k), _ptr(v),
                                        _ptr(beta), _ptr(g_or_a), _ptr(A_log), _ptr(dt_bias),
                                        _ptr(dO), _ptr(M), _ptr(B_or_C), _ptr(ws), ws.numel(),
                                        _stream(dev))
    _check("kda_fragment_summary", st)
    return (M, B_or_C) if mode == KDA_FRAG_FWD else B_or_C


def kda_transfer_walk(doc_frag, M, B, S0=None, *, reverse=False, precision=None, S_in=None,
                      S_final=None, ws=None):
    """Returns (S_in [F,H,d,d], S_final [N,H,d,d]).  precision: a KDA_WALK_* product format
    (default WALK_DEFAULT); ws (optional, >= 256 bytes) receives the device status."""
    F, H, d, _ = M.shape
    N = doc_frag.numel() - 1
    dev = M.device
    if precision is None:
        precision = WALK_DEFAULT
    if S_in is None:
        S_in = torch.empty_like(M)
    if S_final is None:
        S_final = torch.empty((N, H, d, d), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        st = lib().kda_transfer_walk(N, _ptr(doc_frag), F, H, _ptr(M), _ptr(B), _ptr(S0),
                                     int(bool(reverse)), int(precision), _ptr(S_in),
                                     _ptr(S_final), _ptr(ws), _stream(dev))
    _check("kda_transfer_walk", st)
    return S_in, S_final


def make_conv_problem(T, N, C, cu_seqlens=None, *, activation=True, out_dtype=torch.bfloat16):
    if out_dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("out_dtype must be torch.float32 or torch.bfloat16")
    return kda_conv_problem(int(T), int(N), int(C), int(bool(activation)),
                            int(out_dtype == torch.float32),
                            None if cu_seqlens is None else cu_seqlens.data_ptr())


def kda_conv_workspace_size(T, N, C):
    pr = make_conv_problem(T, N, C)
    pr.cu_seqlens = 16  # size queries never read it
    ws = ctypes.c_size_t(0)
    _check("kda_conv_workspace_size", lib().kda_conv_workspace_size(ctypes.byref(pr), ctypes.byref(ws)))
    return ws.value


def _conv_shape(x, cu_seqlens):
    T = x.shape[0]
    C = x.numel() // max(T, 1) if T else int(torch.tensor(x.shape[1:]).prod())
    return T, cu_seqlens.numel() - 1, C


def kda_conv_fwd(x, w, cu_seqlens, *, bias=None, halo=None, activation=True,
                 out_dtype=torch.bfloat16, y=None):
    """Width-4 causal conv1d (+ SiLU) of x [T, ...] (bf16, C channels per token) with taps w
    [C, 4] fp32; halo [N, 3, C] bf16 or None.  Returns y with x's shape in out_dtype."""
    T, N, C = _conv_shape(x, cu_seqlens)
    pr = make_conv_problem(T, N, C, cu_seqlens, activation=activation, out_dtype=out_dtype)
    if y is None:
        y = torch.empty(x.shape, dtype=out_dtype, device=x.device)
    _check_dtypes({"y": y}, out_dtype)
    with torch.cuda.device(x.device):
        st = lib().kda_conv_fwd(ctypes.byref(pr), _ptr(x), _ptr(w), _ptr(bias), _ptr(halo), _ptr(y),
                                _stream(x.device))
    _check("kda_conv_fwd", st)
    return y


def kda_conv_bwd(x, w, cu_seqlens, dy, *, bias=None, halo=None, activation=True, want_dhalo=None,
                 ws=None):
    """Backward of L = sum(y * dy) (dy in y's dtype).  Returns dict dx (dy's dtype, x's shape),
    dw [C, 4], dbias [C] (when bias is given), dhalo [N, 3, C] (when halo is given)."""
    T, N, C = _conv_shape(x, cu_seqlens)
    out_dtype = dy.dtype
    pr = make_conv_problem(T, N, C, cu_seqlens, activation=activation, out_dtype=out_dtype)
    dev = x.device
    if ws is None:
        ws = _empty_bytes(kda_conv_workspace_size(T, N, C), dev)
    out = dict(dx=torch.empty(x.shape, dtype=out_dtype, device=dev),
               dw=torch.empty((C, 4), dtype=torch.float32, device=dev))
    if bias is not None:
        out["dbias"] = torch.empty((C,), dtype=torch.float32, device=dev)
    if halo is not None and want_dhalo is not False:
        out["dhalo"] = torch.empty((N, 3, C), dtype=out_dtype, device=dev)
    with torch.cuda.device(dev):
        st = lib().kda_conv_bwd(ctypes.byref(pr), _ptr(x), _ptr(w), _ptr(bias), _ptr(halo),
                                _ptr(dy), _ptr(out["dx"]), _ptr(out["dw"]), _ptr(out.get("dbias")),
                                _ptr(out.get("dhalo")), _ptr(ws), ws.numel(), _stream(dev))
    _check("kda_conv_bwd", st)
    return out


def kda_read_device_status(ws) -> int:
    v = ctypes.c_int(0)
    with torch.cuda.device(ws.device):
        _check("kda_read_device_status",
               lib().kda_read_device_status(_ptr(ws), ctypes.byref(v), _stream(ws.device)))
    return v.value


def kda_selftest_wait_timeout(ws, limit_us=20000):
    """Runs a kernel whose bounded wait must time out; its KDA_ERR_TIMEOUT lands in ws's status."""
    with torch.cuda.device(ws.device):
        _check("kda_selftest_wait_timeout",
               lib().kda_selftest_wait_timeout(_ptr(ws), ctypes.c_uint32(int(limit_us)), _stream(ws.device)))


def kda_profile_enable(enable=True):
    _check("kda_profile_enable", lib().kda_profile_enable(int(bool(enable))))


def kda_profile_collect():
    """{kernel name: (summed device ms, launches)} since the last collect (waits for events)."""
    n = lib().kda_kernel_count()
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_uint64 * n)()
    _check("kda_profile_collect", lib().kda_profile_collect(ms, cnt))
    return {lib().kda_kernel_name(i).decode(): (ms[i], cnt[i]) for i in range(n)}


def kda_launch_counter() -> int:
    return int(lib().kda_launch_counter())
