"""Host threads calling the library at once.

The C ABI allows calls from several host threads at once, each with its own
workspace; the library's only shared state is a per-device cache of launch
facts filled by the first call.  A fresh interpreter (so that those caches
start empty) runs six threads, released together by a barrier, each on a CUDA
stream of its own: plain verification (bf16 twice, fp32 once), top-k / top-p
filtered verification, draft-side sampling and LM-head-fused verification.
Each thread repeats its call four times; every repeat must give the same
result, and that result must equal the fp64 oracle's (with the usual
exemption band for decisions within 1e-5 of a threshold).
"""
import os
import pickle
import subprocess
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
from speculative_decoding_verification_65_gb300 import synth  # noqa: E402
from tests.parity_util import (BAND, MAX_EXEMPT_FRACTION, check_bound,  # noqa: E402
                               check_invariants, compare)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
NTHREADS = os.cpu_count() or 1
REPEATS = 4

# The child process: loads the jobs, runs one thread per job, writes back the
# outputs of every repeat (or the errors met).
CHILD = r"""
import pickle, sys, threading
import numpy as np
import torch
import speculative_decoding_verification_65_gb300 as sv

jobs = pickle.load(open(sys.argv[1], "rb"))
repeats = int(sys.argv[3])
torch.cuda.set_device(0)
sv.library()
gate = threading.Barrier(len(jobs))
outs, errs = [None] * len(jobs), []


def dev(a):
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(a).cuda()


def call(kind, t):
    if kind == "verify":
        return sv.spec_verify(t["target"], t["draft"], t["tokens"], t["u_accept"],
                              t["u_resample"], t["temperature"])
    if kind == "filtered":
        return sv.spec_verify_filtered(t["target"], t["draft"], t["tokens"], t["u_accept"],
                                       t["u_resample"], t["temperature"], top_k=t["top_k"],
                                       top_p=t["top_p"])
    if kind == "sample":
        return (sv.spec_sample(t["logits"], t["u"], t["temperature"]),)
    return sv.spec_verify_lmhead(t["hidden"], t["lm_head"], t["draft"], t["tokens"],
                                 t["u_accept"], t["u_resample"], t["temperature"])


def work(i):
    kind, arrays = jobs[i]
    try:
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            t = {n: dev(a) for n, a in arrays.items()}
            s.synchronize()
            gate.wait(timeout=300)
            res = [call(kind, t) for _ in range(repeats)]
            s.synchronize()
        outs[i] = [[x.cpu().numpy() for x in r] for r in res]
    except BaseException as e:
        errs.append(f"job {i} ({kind}): {e!r}")
        gate.abort()


threads = [threading.Thread(target=work, args=(i,)) for i in range(len(jobs))]
for th in threads:
    th.start()
for th in threads:
    th.join()
pickle.dump((outs, errs), open(sys.argv[2], "wb"))
"""


def _verify_arrays(c, **extra):
    return dict(target=c.target, draft=c.draft, tokens=c.tokens, u_accept=c.u_accept,
                u_resample=c.u_resample, temperature=c.temperature, **extra)


def _jobs():
    v1 = synth.make_config(2, seed_offset=0)         # B32 k5 V32000 bf16
    v2 = synth.make_config(2, seed_offset=7)
    v3 = synth.make_config(1)                        # B4 k4 V1024 fp32
    f = synth.make_config(1, B=12, seed_offset=3)
    f.tokens = np.argmax(synth.decode(f.draft), axis=2).astype(np.int32)  # kept by any filter
    tk = np.array([0, 1, 5, 10, 50, 1000] * 2, np.int32)
    tp = np.array([1.0, 0.5, 0.9, 0.99] * 3, np.float32)
    sc = synth.make_sample_config(2)
    lc = synth.make_lmhead_case(B=8, k=3, V=600, d=128, dtype="bf16", recipe="grid", seed=21,
                                T=(0.0, 1.0))
    cases = [("verify", v1), ("verify", v2), ("verify", v3), ("filtered", (f, tk, tp)),
             ("sample", sc), ("lmhead", lc)]
    jobs = []
    for kind, c in cases:
        if kind == "verify":
            jobs.append((kind, _verify_arrays(c)))
        elif kind == "filtered":
            jobs.append((kind, _verify_arrays(c[0], top_k=c[1], top_p=c[2])))
        elif kind == "sample":
            jobs.append((kind, dict(logits=c.logits, u=c.u, temperature=c.temperature)))
        else:
            jobs.append((kind, dict(hidden=c.hidden, lm_head=c.lm_head, draft=c.draft,
                                    tokens=c.tokens, u_accept=c.u_accept,
                                    u_resample=c.u_resample, temperature=c.temperature)))
    return cases, jobs


def _check_sample(sc, g):
    r, tr = oracle.sample(sc.logits, sc.u.astype(np.float64), sc.temperature.astype(np.float64),
                          nthreads=NTHREADS)
    exempt = 0
    for i in np.nonzero(g != r)[0]:
        assert sc.temperature[i] > 0 and r[i] >= 0 and g[i] >= 0, (i, g[i], r[i])
        margin = min(float(sc.u[i]) - tr[i, 0], tr[i, 1] - float(sc.u[i]))
        assert margin < BAND, (i, g[i], r[i], margin)
        exempt += 1
    assert exempt <= MAX_EXEMPT_FRACTION * len(r), exempt


def _check_filtered(c, tk, tp, gt, gn):
    rt, rn, tr = oracle.verify_filtered(c.target, c.draft, c.tokens, c.u_accept, c.u_resample,
                                        c.temperature, tk, tp, nthreads=NTHREADS)
    near = np.nan_to_num(tr[:, c.k + 3], nan=1.0) < BAND   # top-p cut within the band
    keep = np.nonzero(~near)[0]
    sub = c.subset(keep)
    sub.tokens = c.tokens[keep]
    rep = compare(sub, gt[keep], gn[keep], rt[keep], rn[keep], tr[keep][:, :c.k + 3])
    check_bound(rep)
    cut = int(np.sum(near & ((gn != rn) | np.any(gt != rt, axis=1))))
    assert cut <= max(1, MAX_EXEMPT_FRACTION * rep["decisions"]), cut


def test_concurrent_first_calls_from_host_threads(tmp_path):
    cases, jobs = _jobs()
    src, dst = tmp_path / "jobs.pkl", tmp_path / "outs.pkl"
    with open(src, "wb") as fh:
        pickle.dump(jobs, fh)
    env = dict(os.environ, PYTHONPATH=ROOT + os.pathsep + os.environ.get("PYTHONPATH", ""))
    run = subprocess.run([sys.executable, "-c", CHILD, str(src), str(dst), str(REPEATS)],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert run.returncode == 0, run.stderr[-3000:]
    with open(dst, "rb") as fh:
        outs, errs = pickle.load(fh)
    assert not errs, errs
    for (kind, c), res in zip(cases, outs):
        assert res is not None and len(res) == REPEATS, kind
        for r in res[1:]:  # every repeat on the thread's own workspace agrees
            assert all(np.array_equal(a, b) for a, b in zip(res[0], r)), kind
        out = res[0]
        if kind == "verify":
            rt, rn, tr = oracle.verify(c.target, c.draft, c.tokens, c.u_accept, c.u_resample,
                                       c.temperature, nthreads=NTHREADS)
            check_invariants(c, out[0], out[1])
            rep = compare(c, out[0], out[1], rt, rn, tr)
            check_bound(rep)
        elif kind == "filtered":
            f, tk, tp = c
            _check_filtered(f, tk, tp, out[0], out[1])
        elif kind == "sample":
            _check_sample(c, out[0])
        else:
            rt, rn, tr = oracle.verify_lmhead(c.hidden, c.lm_head, c.draft, c.tokens,
                                              c.u_accept, c.u_resample, c.temperature,
                                              nthreads=NTHREADS)
            check_invariants(c, out[0], out[1])
            rep = compare(c, out[0], out[1], rt, rn, tr)
            check_bound(rep)  # grid inputs: the logits are exact in fp32
