"""Builds the in-tree CUDA library libkda_gb300.so for sm_103a (nvcc, one -gencode, parallel TUs)."""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libkda_gb300.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC = os.environ.get("NVCC", "nvcc")
# -ftz=true: single-precision results below 2^-126 flush to zero.  The kernels' exponentials of
# gate differences then compile to a multiply and one ex2 (no subnormal rescaling around it); the
# only values affected lie below 1.2e-38, far under every error bound.
CODEGEN = ["-O3", "-lineinfo", "-std=c++17", "-ftz=true"]
FLAGS = CODEGEN + ["-Xcompiler", "-fPIC", "-Xcompiler", "-Wall", "--expt-relaxed-constexpr", "-I",
                   os.path.join(ROOT, "include")]


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.cuh"))
            + glob.glob(os.path.join(ROOT, "include", "*.h")))


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile every csrc/*.cu for sm_103a and link libkda_gb300.so; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    deps = _deps()
    if not force and not _stale(LIB, deps):
        return LIB
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        cmd = [NVCC, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        results = list(ex.map(compile_one, _sources()))
    if verbose or ptxas_info:
        for _, err in results:
            if err:
                print(err)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [NVCC, *ARCH, "-shared", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB



def _code_only(text: str) -> str:
    """C / C++ / CUDA source without its comments, trailing blanks and empty lines (string and
    character literals are kept as written)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":  # literal: copy through the closing quote, honouring escapes
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    lines = (line.rstrip() for line in "".join(out).splitlines())
    return "\n".join(line for line in lines if line)


# the translation unit of each profiled kernel (bench.py stage labels)
KERNEL_SOURCES = {
    "k_intra_fwd": "kda_intra.cu",
    "k_chain_fwd": "kda_chain_tc.cu",
    "k_chain_bwd": "kda_chain_tc.cu",
    "k_bwd_gemms_tc": "kda_bwd_tc.cu",
    "k_bwd_intra": "kda_bwd.cu",
}


def source_digest(kernel: str = None) -> str:
    """Short digest of the code of the CUDA sources and the ABI header, comments left out, and of
    the code generation flags (ties profiles to the code they measured; a comment-only edit keeps
    the digest).  With a kernel
    label: only that kernel's translation unit, the launch code (kda_api.cu), the shared headers
    and the ABI header, so a change to another kernel keeps this one's measurements."""
    import hashlib
    deps = _deps()
    if kernel is not None:
        own = {KERNEL_SOURCES[kernel], "kda_api.cu"}
        deps = [d for d in deps if not d.endswith(".cu") or os.path.basename(d) in own]
    h = hashlib.sha256()
    h.update(" ".join(ARCH + CODEGEN).encode())
    for path in sorted(deps):
        h.update(os.path.basename(path).encode())
        with open(path, encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
