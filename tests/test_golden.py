"""Stored oracle fixture: input-generator determinism and oracle stability."""
import os

import numpy as np

import oracle
from tiled_attention_forward_fa2_gb300.inputs import WORKLOADS

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load():
    rows, lse, o, sha = [], [], [], None
    with open(os.path.join(HERE, "b1h1n256d64_rows.txt")) as f:
        for line in f:
            if line.startswith("#"):
                continue
            parts = line.split()
            if parts[0] == "sha256_qkv":
                sha = parts[1]
            elif parts[0] == "row":
                rows.append(int(parts[1]))
                lse.append(float(parts[3]))
                o.append([float(x) for x in parts[5:]])
    return sha, np.array(rows), np.array(lse), np.array(o)


def test_golden_inputs_and_oracle():
    import importlib.util
    spec = importlib.util.spec_from_file_location("make_golden", os.path.join(HERE, "make_golden.py"))
    mg = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mg)
    sha, rows, lse, o = _load()
    w = WORKLOADS["b1h1n256d64"]
    q, k, v = w.qkv()
    assert mg.digest(q, k, v) == sha, "seeded input generator changed its output"
    o2, lse2 = oracle.attn_rows(q, k, v, w.causal, w.scale, np.zeros(len(rows), np.int64), rows)
    assert np.max(np.abs(o2 - o)) <= 1e-12 and np.max(np.abs(lse2 - lse)) <= 1e-12
