"""The code digest that ties committed ncu figures to the kernels they measured (CPU only)."""
import os
import shutil

import pytest

from linear_attention_chunked_gb300 import build


def test_code_only_drops_comments_and_blank_lines_but_keeps_literals():
    src = ('int a = 1;  // trailing\n'
           '/* block\n   comment */\n'
           '\n'
           'const char* s = "// not a comment /* nor this */";\n'
           "char c = '/'; char e = '\\'';\n"
           'asm volatile("mov.b32 %0, %1;\\n" : "=r"(x) : "r"(y));  /* tail */\n')
    out = build._code_only(src)
    assert out.splitlines() == [
        'int a = 1;',
        'const char* s = "// not a comment /* nor this */";',
        "char c = '/'; char e = '\\'';",
        'asm volatile("mov.b32 %0, %1;\\n" : "=r"(x) : "r"(y));',
    ]


@pytest.fixture
def tree(tmp_path, monkeypatch):
    """A copy of the CUDA sources and the ABI header that the digest functions read instead."""
    csrc = tmp_path / "csrc"
    inc = tmp_path / "include"
    shutil.copytree(build.CSRC, csrc)
    shutil.copytree(os.path.join(build.ROOT, "include"), inc)
    monkeypatch.setattr(build, "CSRC", str(csrc))
    monkeypatch.setattr(build, "ROOT", str(tmp_path))
    return csrc


def _edit(path, fn):
    with open(path) as f:
        text = f.read()
    with open(path, "w") as f:
        f.write(fn(text))


def test_comment_edit_keeps_every_digest(tree):
    before = {k: build.source_digest(k) for k in build.KERNEL_SOURCES}
    whole = build.source_digest()
    _edit(tree / "kda_bwd.cu", lambda t: "// a new note\n" + t.replace("\n", "\n\n", 3))
    assert build.source_digest() == whole
    assert {k: build.source_digest(k) for k in build.KERNEL_SOURCES} == before


def test_code_edit_changes_only_its_kernels_digest(tree):
    before = {k: build.source_digest(k) for k in build.KERNEL_SOURCES}
    whole = build.source_digest()
    _edit(tree / "kda_intra.cu", lambda t: t + "\nnamespace kda { int unused_marker = 1; }\n")
    after = {k: build.source_digest(k) for k in build.KERNEL_SOURCES}
    assert build.source_digest() != whole
    assert after["k_intra_fwd"] != before["k_intra_fwd"]
    for k in build.KERNEL_SOURCES:
        if k != "k_intra_fwd":
            assert after[k] == before[k], k


def test_shared_header_edit_changes_every_kernels_digest(tree):
    before = {k: build.source_digest(k) for k in build.KERNEL_SOURCES}
    _edit(tree / "kda_internal.cuh", lambda t: t + "\nconstexpr int kUnusedMarker = 2;\n")
    after = {k: build.source_digest(k) for k in build.KERNEL_SOURCES}
    assert all(after[k] != before[k] for k in build.KERNEL_SOURCES)


def test_every_profiled_kernel_names_an_existing_source():
    for k, f in build.KERNEL_SOURCES.items():
        assert os.path.exists(os.path.join(build.CSRC, f)), (k, f)
