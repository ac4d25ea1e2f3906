"""Pins for the in-seq-split comparator (no GPU)."""
import numpy as np

from conftest import GOLDEN
from oracle import inseq


def _cases():
    cases, cur = [], None
    with open(f"{GOLDEN}/inseq_examples.txt", encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("case"):
                tok = line.split()
                cur = {"lengths": [int(v) for v in tok[3].split(",")], "sp": int(tok[5]),
                       "gran": int(tok[7]) if len(tok) > 7 else 1, "expect": []}
                cases.append(cur)
            else:
                k, v = line.split(":")
                k = k.split()
                cur["expect"].append((int(k[1]), int(k[3]), v.split()))
    return cases


def test_page_examples():
    for case in _cases():
        for rank, req, v in case["expect"]:
            p = inseq.in_seq_positions(case["lengths"][req], case["sp"], rank, case["gran"])
            if v == ["empty"]:
                assert len(p) == 0
            else:
                assert p[0] == int(v[0]) and p[-1] == int(v[1]) and len(p) == int(v[1]) - int(v[0]) + 1


def test_in_seq_partitions_each_request():
    rng = np.random.default_rng(0)
    lengths = rng.integers(1, 300, 9).tolist()
    for sp in (1, 3, 8):
        for gran in (1, 64):
            seen = [np.zeros(L, dtype=int) for L in lengths]
            for r in range(sp):
                bid, pos = inseq.in_seq_split(lengths, sp, r, gran)
                for b, p in zip(bid, pos):
                    seen[b][p] += 1
            assert all(np.all(s == 1) for s in seen)


def test_causal_pairs():
    assert inseq.causal_pairs(np.array([0, 1, 5])) == 1 + 2 + 6
