"""Host-side pieces of bench.py that the reported figures depend on: the
FLOP count of the prefill workloads (legal pairs, against the oracle's own
enumeration) and the kernel-source hashes that keep stale ncu traffic out of
the JSON line.  CPU only."""
import os
import sys

import numpy as np

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_legal_pairs_match_the_oracle():
    g = np.random.default_rng(11)
    cases = [(64, 128, 0), (4096, 4096, 0), (1, 2053, 0), (512, 4096, 1024), (7, 3, 0),
             (0, 5, 0), (5, 0, 0), (300, 40, 0), (100, 1000, 1)]
    cases += [(int(g.integers(0, 300)), int(g.integers(0, 300)), int(g.integers(0, 50)))
              for _ in range(20)]
    for Qb, Kb, w in cases:
        assert bench.legal_pairs(Qb, Kb, w) == oracle.legal_pairs(Qb, Kb, w), (Qb, Kb, w)


def test_headline_flop_count():
    # B=4 Hq=32 Q=K=4096 D=Dv=128: 4096 * 4097 / 2 pairs per head, 512 FLOP a pair
    P = bench.PREFILL
    flop = P["B"] * P["Hq"] * bench.legal_pairs(P["Q"], P["K"]) * (2 * P["D"] + 2 * P["Dv"])
    assert flop == 549_890_031_616


def test_source_hashes_cover_every_kernel_source():
    for name, rel in bench.KERNEL_SOURCES.items():
        paths = (rel,) if isinstance(rel, str) else rel
        for r in paths:
            assert os.path.exists(os.path.join(ROOT, r)), (name, r)
        h = bench.source_sha(rel)
        assert len(h) == 16 and int(h, 16) >= 0
    # the backward's hash changes with either of its two files
    assert bench.source_sha(bench.KERNEL_SOURCES["backward"]) != bench.source_sha(
        bench.KERNEL_SOURCES["backward"][0])
