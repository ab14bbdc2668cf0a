"""The index arithmetic every kernel shares (csrc/common.cuh), compiled for
the host and checked against the legal-key mask built from numpy's triangle
routines (the same construction that pins the oracle):

* legal_range(q) is exactly the set of keys row q may attend to, for both
  causal masks, no mask, windows, Q > K and Q < K;
* rows_for_keys(k0, k1) is exactly the set of rows with a legal key in
  [k0, k1) -- the row range the dK/dV kernels walk for a tile of keys.

CPU only (nvcc compiles the host program; no GPU is touched)."""
import os
import shutil
import subprocess

import numpy as np
import pytest

from tests.oracle_pins import mask_matrix

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "causal_gqa_attention_online_gb300", "csrc")

PROGRAM = r'''
#include <cstdio>
#include "common.cuh"
int main() {
    int Qb, Kb, window, mask, blk;
    while (std::scanf("%d %d %d %d %d", &Qb, &Kb, &window, &mask, &blk) == 5) {
        for (int q = 0; q < Qb; ++q) {
            int lo, hi;
            attn::legal_range(q, Qb, Kb, window, mask, lo, hi);
            std::printf("%d %d ", lo, hi);
        }
        std::printf("\n");
        for (int k0 = 0; k0 < Kb; k0 += blk) {
            const int k1 = k0 + blk < Kb ? k0 + blk : Kb;
            int qf, qe;
            attn::rows_for_keys(k0, k1, Qb, Kb, window, mask, qf, qe);
            std::printf("%d %d ", qf, qe);
        }
        std::printf("\n");
    }
    return 0;
}
'''


@pytest.fixture(scope="module")
def index_prog(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    d = tmp_path_factory.mktemp("idx")
    src = d / "idx.cu"
    src.write_text(PROGRAM)
    exe = d / "idx"
    r = subprocess.run([nvcc, "-std=c++17", "-I", CSRC, "-o", str(exe), str(src)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return str(exe)


def cases():
    g = np.random.default_rng(21)
    out = [(5, 9, 0, 0, 3), (9, 5, 0, 0, 2), (7, 7, 3, 0, 4), (6, 10, 0, 1, 3), (6, 10, 4, 1, 5),
           (8, 4, 0, 2, 3), (1, 2053, 0, 0, 64), (1, 2053, 700, 0, 64), (64, 128, 0, 0, 32)]
    for _ in range(60):
        Qb, Kb = int(g.integers(1, 90)), int(g.integers(1, 90))
        mask = int(g.integers(0, 3))
        window = 0 if mask == 2 or g.random() < 0.4 else int(g.integers(1, 40))
        out.append((Qb, Kb, window, mask, int(g.integers(1, 40))))
    return out


def test_legal_range_and_rows_for_keys(index_prog):
    cs = cases()
    inp = "".join(f"{Qb} {Kb} {w} {m} {blk}\n" for Qb, Kb, w, m, blk in cs)
    r = subprocess.run([index_prog], input=inp, capture_output=True, text=True, timeout=60)
    assert r.returncode == 0
    lines = r.stdout.splitlines()
    assert len(lines) == 2 * len(cs)
    for i, (Qb, Kb, w, m, blk) in enumerate(cs):
        mm = mask_matrix(Qb, Kb, w, m)
        ranges = np.array(lines[2 * i].split(), dtype=np.int64).reshape(Qb, 2)
        for q in range(Qb):
            lo, hi = ranges[q]
            keys = np.flatnonzero(mm[q])
            if keys.size == 0:
                assert hi <= lo or hi <= 0, (Qb, Kb, w, m, q, lo, hi)
            else:
                assert (lo, hi) == (keys[0], keys[-1] + 1), (Qb, Kb, w, m, q, lo, hi)
                assert keys.size == hi - lo  # an interval
        blocks = np.array(lines[2 * i + 1].split(), dtype=np.int64).reshape(-1, 2)
        for bi, k0 in enumerate(range(0, Kb, blk)):
            k1 = min(k0 + blk, Kb)
            qf, qe = blocks[bi]
            rows = np.flatnonzero(mm[:, k0:k1].any(axis=1))
            got = set(range(max(qf, 0), min(qe, Qb)))
            assert got == set(rows.tolist()), (Qb, Kb, w, m, k0, k1, qf, qe)
