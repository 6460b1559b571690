"""Rules on the kernel sources that need no GPU.

The kernels read only this GPU's own memory: no TMA copy (cp.async.bulk...)
uses cluster multicast.  The one `multicast::cluster` in the sources is
tcgen05.commit's arrive on both CTAs' barriers of an SM pair, which moves no
data.
"""
from __future__ import annotations

import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "warp_specialized_tma_gb300", "csrc")


def _sources():
    for name in sorted(os.listdir(CSRC)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(CSRC, name)) as fh:
                yield name, fh.read()


def test_no_tma_multicast_copy():
    for name, text in _sources():
        for m in re.finditer(r"cp\.(?:reduce\.)?async\.bulk[^\"]*", text):
            assert "multicast" not in m.group(0), f"{name}: {m.group(0)}"


def test_multicast_only_in_the_pair_commit():
    hits = [(name, line.strip()) for name, text in _sources() for line in text.splitlines() if "multicast" in line
            and not line.strip().startswith("//")]
    assert hits, "the SM-pair commit is expected to multicast its arrive"
    for name, line in hits:
        assert "tcgen05.commit" in line, f"{name}: {line}"
