"""The oracle and the CUDA path share no code, and the product never reaches
the oracle (CPU, static checks of the sources)."""
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "gated_deltanet_recurrence_gdn_gb300")
ORACLE = os.path.join(ROOT, "oracle")
SYNTH = os.path.join(ROOT, "synth")
CODE = (".py", ".cu", ".cuh", ".h", ".c", ".cpp", ".sh")
SKIP_DIRS = {"_build", "__pycache__"}
# everything committed that holds code: the package, the oracle, the input
# generators, the tests and the entry scripts at the top
COMMITTED = [PKG, ORACLE, SYNTH, os.path.join(ROOT, "tests"), os.path.join(ROOT, "include"),
             os.path.join(ROOT, "bench.py"), os.path.join(ROOT, "__graft_entry__.py")]


def _sources(top):
    if os.path.isfile(top):
        yield top, open(top, encoding="utf-8", errors="replace").read()
        return
    for d, dirs, files in os.walk(top):
        dirs[:] = [x for x in dirs if x not in SKIP_DIRS]
        for f in files:
            if f.endswith(CODE):
                p = os.path.join(d, f)
                yield p, open(p, encoding="utf-8", errors="replace").read()


def _imports(src, module):
    pat = r"^\s*(import\s+%s\b|from\s+%s\b)" % (module, module)
    return re.search(pat, src, flags=re.M) is not None


def test_product_never_reaches_the_oracle():
    for p, src in _sources(PKG):
        assert not _imports(src, "oracle"), p
        assert "gdn_oracle" not in src, p
        assert not re.search(r'#\s*include\s*[<"][^>"]*oracle', src), p


def test_oracle_never_reaches_the_product():
    for p, src in _sources(ORACLE):
        assert not _imports(src, "gated_deltanet_recurrence_gdn_gb300"), p
        assert not _imports(src, "synth"), p
        # no CUDA-path header, helper or kernel file is pulled in
        for inc in re.findall(r'#\s*include\s*[<"]([^>"]+)[>"]', src):
            assert inc in {"math.h", "stddef.h", "stdlib.h", "string.h", "stdint.h"}, (p, inc)
        assert "csrc" not in src, p


def test_input_generators_import_neither_side():
    for p, src in _sources(SYNTH):
        assert not _imports(src, "oracle"), p
        assert not _imports(src, "gated_deltanet_recurrence_gdn_gb300"), p


def test_no_committed_code_uses_scratch_folder():
    me = os.path.abspath(__file__)
    for top in COMMITTED:
        for p, src in _sources(top):
            if os.path.abspath(p) == me:
                continue
            assert not re.search(r"(?<![A-Za-z0-9])_work/", src), p
