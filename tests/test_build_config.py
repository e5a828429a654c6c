"""The build configuration and the tree's text hygiene (no GPU needed).

The pages' change carries a build-config unit test and a whitespace check
("vLLM: integrate FP16 packed QSA extension", Validation); these are the
counterparts here: the library is compiled for sm_103a only, optimised, with
the CUDA runtime linked in; the oracle without fast-math or FMA contraction
(its binary32 and binary64 arithmetic is the reference); and no source,
test, header or note carries trailing whitespace, a blank line at its end
or a merge-conflict marker."""
import os
import re

from sparse_paged_attention_qsa_gb300 import build as qbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_library_is_built_for_sm_103a_only():
    assert qbuild.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert "-O3" in qbuild.NVCC_FLAGS
    assert not any("fast_math" in f or "fast-math" in f for f in qbuild.NVCC_FLAGS)
    src = open(qbuild.__file__).read()
    assert '"-cudart", "static"' in src            # no runtime to find at load time
    assert "-maxrregcount" not in src              # register caps live in the kernels


def test_oracle_is_built_without_fast_math_or_contraction():
    src = open(os.path.join(ROOT, "oracle", "__init__.py")).read()
    assert "-ffp-contract=off" in src and "-fno-fast-math" in src
    assert "-ffast-math" not in src and "-Ofast" not in src


def _text_files():
    dirs = ["include", "oracle", "sparse_paged_attention_qsa_gb300", "tests", "profiles"]
    exts = (".py", ".c", ".h", ".cu", ".cuh", ".md", ".txt", ".json")
    for d in dirs:
        for base, subdirs, files in os.walk(os.path.join(ROOT, d)):
            subdirs[:] = [s for s in subdirs if s not in ("_build", "__pycache__", "golden")]
            for f in files:
                if f.endswith(exts):
                    yield os.path.join(base, f)
    for f in ("README.md", "DESIGN.md", "bench.py", "__graft_entry__.py"):
        yield os.path.join(ROOT, f)


def test_no_trailing_whitespace_or_conflict_markers():
    bad = []
    marker = re.compile(r"^(<<<<<<<|=======$|>>>>>>>)")
    for path in _text_files():
        text = open(path, encoding="utf-8").read()
        rel = os.path.relpath(path, ROOT)
        for n, line in enumerate(text.split("\n"), 1):
            if line != line.rstrip(" \t"):
                bad.append(f"{rel}:{n}: trailing whitespace")
            if marker.match(line):
                bad.append(f"{rel}:{n}: conflict marker")
        if text.endswith("\n\n"):
            bad.append(f"{rel}: blank line at end of file")
    assert not bad, "\n".join(bad[:20])
