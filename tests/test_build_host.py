"""The build covers every source: each file under csrc/ is either compiled (SOURCES) or a
header whose changes make the library stale (HEADERS), and each public header is an input
of the staleness check."""
import os

from rmsnorm_fwd_02_gb300 import build as B


def test_every_csrc_file_is_compiled_or_tracked():
    files = set(os.listdir(B.CSRC))
    assert files == set(B.SOURCES) | set(B.HEADERS), files ^ (set(B.SOURCES) | set(B.HEADERS))


def test_public_headers_are_build_inputs():
    inputs = {os.path.basename(p) for p in B._inputs()}
    for h in os.listdir(os.path.join(B.ROOT, "include")):
        assert h in inputs, h
