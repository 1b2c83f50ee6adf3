"""FP64 CPU oracle of the width-4 causal depthwise conv1d + SiLU that feeds KDA's q, k and v
(test infrastructure only: the same import rules as the rest of this package apply).

Source: the KCP transfer-walk page (flashinfer PR #7176), PR description: the module forward
("B1") runs the conv halo exchange, the conv and the KDA state passing and recurrence, and the
kernel family ships a width-4 causal conv1d + SiLU training backend with a halo variant.  The
pages print no formula; this is the plainest reading of "width-4 causal conv1d + SiLU" on packed
documents, and it is the one the library implements:

    z[t, c] = b[c] + sum_{j=0..3} w[c, j] * x[t - 3 + j, c]      (depthwise over channels c)
    y[t, c] = silu(z[t, c]) = z[t, c] * sigmoid(z[t, c])

inside each document of the pack (cu_seqlens).  A position t - 3 + j before the document's first
token reads the document's halo row (halo[n, 3 + (t - 3 + j - start), c]: the three tokens that
precede the document, e.g. the end of the previous fragment of the same long document), or zero
when no halo is given.  The backward of L = sum(y * dy) is

    dz = dy * silu'(z),   silu'(z) = s (1 + z (1 - s)),  s = sigmoid(z)
    dx[t', c] = sum_j w[c, j] dz[t' + 3 - j, c]   (t' + 3 - j inside the same document)
    dw[c, j] = sum_t dz[t, c] x[t - 3 + j, c],   db[c] = sum_t dz[t, c],
    dhalo[n, i, c] = sum over the document's first tokens of w[c, j] dz[t, c] where t - 3 + j
                     addresses halo row i.

Parity status: pinned by tests/test_conv_pins.py -- the identity tap against SiLU written with
scipy's logistic function, a pure three-token shift (causality and the document reset), every
channel against numpy.convolve, the halo split invariance (a document cut in two with the first
piece's last three tokens as the second's halo), and central finite differences of every
gradient (x, w, b, halo).
"""
from __future__ import annotations

import numpy as np

WIDTH = 4


def _sigmoid(z):
    # numerically safe logistic function for either sign of z
    e = np.exp(-np.abs(z))
    return np.where(z >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


def _docs(cu_seqlens):
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    return [(int(cu[n]), int(cu[n + 1])) for n in range(len(cu) - 1)]


def _padded(x, a, e, halo_n):
    """The document's rows with the three rows before it (halo or zeros) in front."""
    C = x.shape[1]
    xp = np.zeros((e - a + WIDTH - 1, C))
    if halo_n is not None:
        xp[:WIDTH - 1] = halo_n
    xp[WIDTH - 1:] = x[a:e]
    return xp


def conv_fwd(x, w, cu_seqlens, bias=None, halo=None, activation=True):
    """x [T, C], w [C, 4], bias [C] or None, halo [N, 3, C] or None.  Returns (y, z)."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    T, C = x.shape
    z = np.zeros((T, C))
    for n, (a, e) in enumerate(_docs(cu_seqlens)):
        xp = _padded(x, a, e, None if halo is None else np.asarray(halo, np.float64)[n])
        for t in range(e - a):
            acc = np.zeros(C) if bias is None else np.array(bias, dtype=np.float64)
            for j in range(WIDTH):
                acc = acc + w[:, j] * xp[t + j]  # xp[t + j] = x[t - 3 + j]
            z[a + t] = acc
    y = z * _sigmoid(z) if activation else z.copy()
    return y, z


def conv_bwd(x, w, cu_seqlens, dy, bias=None, halo=None, activation=True):
    """Gradients of L = sum(y * dy).  Returns dict dx [T, C], dw [C, 4], db [C], dhalo [N, 3, C]
    (dhalo only when a halo is given)."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    _, z = conv_fwd(x, w, cu_seqlens, bias, halo, activation)
    if activation:
        s = _sigmoid(z)
        dz = dy * s * (1.0 + z * (1.0 - s))
    else:
        dz = dy.copy()
    T, C = x.shape
    docs = _docs(cu_seqlens)
    dx = np.zeros((T, C))
    dw = np.zeros((C, WIDTH))
    dhalo = np.zeros((len(docs), WIDTH - 1, C)) if halo is not None else None
    for n, (a, e) in enumerate(docs):
        xp = _padded(x, a, e, None if halo is None else np.asarray(halo, np.float64)[n])
        for t in range(e - a):
            for j in range(WIDTH):
                dw[:, j] += dz[a + t] * xp[t + j]
                src = t + j - (WIDTH - 1)  # position of the read inside the document
                if src >= 0:
                    dx[a + src] += w[:, j] * dz[a + t]
                elif dhalo is not None:
                    dhalo[n, src + WIDTH - 1] += w[:, j] * dz[a + t]
    out = dict(dx=dx, dw=dw, db=dz.sum(axis=0))
    if dhalo is not None:
        out["dhalo"] = dhalo
    return out
