"""The benchmark's reference-arm JSON line, on the CPU.

`bench.py --impl reference` times the fp64 oracle on the host cores and
prints one JSON line.  For the verify, filtered, sample and tree ops on
their smallest workload, the line must carry every key of the benchmark's
contract: the metric and its unit, the steps and warm-up it ran, a
`cpu_baseline` that describes the same run, and an `e2e` object with no host
copies.  (The LM-head arm draws a 1 GB weight matrix and is left to the
benchmark itself.)
"""
import io
import json
import sys
from contextlib import redirect_stdout

import pytest

from tests.conftest import ROOT

sys.path.insert(0, ROOT)
import bench  # noqa: E402

KEYS = {"impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
        "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
        "cpu_baseline", "e2e"}


@pytest.mark.parametrize("op,metric", [("verify", bench.METRIC), ("filtered", bench.METRIC),
                                       ("sample", bench.SAMPLE_METRIC),
                                       ("tree", bench.TREE_METRIC)])
def test_reference_line(op, metric, monkeypatch):
    for var in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(var, raising=False)
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--op", op,
                                      "--config", "1", "--tree-config", "1", "--steps", "2",
                                      "--warmup", "3", "--cpu-budget", "5"])
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main()
    lines = buf.getvalue().strip().splitlines()
    assert len(lines) == 1, lines
    d = json.loads(lines[0])
    assert KEYS <= d.keys(), KEYS - d.keys()
    assert d["impl"] == "reference" and d["metric"] == metric
    assert d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 3
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["scaling"] == "weak" and d["vs_baseline"] is None and d["data"] == "synthetic"
    assert d["config"]["workload"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"]
    assert cb["value"] == d["value"] and cb["unit"] == d["unit"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


@pytest.mark.parametrize("cfg,B,V", [(1, None, None), (4, 12, 2048)])
def test_oracle_alpha_is_the_overlap_of_p_and_q(cfg, B, V):
    """The verify line's analytic acceptance: the mean over drafted positions
    of the sampling sequences of sum_x min(p, q), against scipy's softmax."""
    import numpy as np
    from scipy import special
    from speculative_decoding_verification_65_gb300 import synth
    case = synth.make_config(cfg, B=B, V=V)
    a, n = bench.oracle_alpha(case, 16)
    seqs = np.flatnonzero(case.temperature > 0)[:16]
    assert n == len(seqs) * case.k
    t, d = synth.decode(case.target), synth.decode(case.draft)
    want = [np.minimum(special.softmax(t[b, i].astype(np.float64) / case.temperature[b]),
                       special.softmax(d[b, i].astype(np.float64) / case.temperature[b])).sum()
            for b in seqs for i in range(case.k)]
    assert abs(a - float(np.mean(want))) < 1e-12
