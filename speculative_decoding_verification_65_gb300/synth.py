"""Seeded synthetic inputs for speculative-sampling verification.

This module is the one piece shared by the CUDA path's tests/bench and the
oracle: it only draws random numbers (numpy PCG64) and holds none of the
verification arithmetic (no softmax, ratio, residual or inverse-CDF).  Draft
tokens are sampled from softmax(d/T) by the Gumbel-max construction
(argmax of d/T + Gumbel noise, written as d/T - log(E), E ~ Exp(1)), which
needs no probabilities at all; greedy (T = 0) sequences take argmax d.

There is no public dataset for this step and no model weights here, so the
workloads below stand in for real language-model logits.  Their shapes and
value distributions follow the five workloads the verification kernel is
specified against:

  1  B=4,    k=4, V=1024,   fp32  gaussian: d ~ N(0,3^2), t = d + N(0,0.7^2)
  2  B=32,   k=5, V=32000,  bf16  gaussian N(0,2^2) with 50 "peak" ids +6,
                                  t = d + N(0,0.5^2), T = 1
  3  B=64,   k=4, V=128256, bf16  Zipf logits -1.1 ln(rank) + N(0,0.3^2) over a
                                  random permutation; the target keeps 51 of
                                  the draft's top-64 ids; T = 0.7
  4  B=256,  k=8, V=151936, fp32  d ~ N(0,2.5^2), t = d + N(0,1); per-sequence
                                  T drawn from {0, 0.5, 1.0, 1.3}
  5  B=1024, k=4, V=128256, bf16  three classes by b mod 3: target == draft
                                  (bit-identical), disjoint peak sets, and
                                  t = d + N(0,0.5^2); T = 1

The bonus target row (position k+1) has no draft row; it is drawn fresh by the
same recipe as the target rows.  bf16 values are generated in fp32 and rounded
to nearest-even; everyone (kernel, oracle, token sampler) reads the rounded
values.  Each sequence has its own child generator (SeedSequence.spawn), so
generation is parallel over sequences and the bytes do not depend on the
thread count.  Seeds: logits 1000*cfg + 0, tokens + 1, uniforms and
temperatures + 2.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

F32 = "f32"
BF16 = "bf16"

CONFIGS = {
    1: dict(B=4, k=4, V=1024, dtype=F32, recipe="gauss", sigma_d=3.0, sigma_n=0.7,
            temps=(1.0,)),
    2: dict(B=32, k=5, V=32000, dtype=BF16, recipe="peaks", sigma_d=2.0, n_peaks=50,
            peak=6.0, sigma_n=0.5, temps=(1.0,)),
    3: dict(B=64, k=4, V=128256, dtype=BF16, recipe="zipf", zipf_s=1.1, sigma_z=0.3,
            top=64, share=0.8, temps=(0.7,)),
    4: dict(B=256, k=8, V=151936, dtype=F32, recipe="gauss", sigma_d=2.5, sigma_n=1.0,
            temps=(0.0, 0.5, 1.0, 1.3)),
    5: dict(B=1024, k=4, V=128256, dtype=BF16, recipe="classes", sigma_d=2.0, n_peaks=50,
            peak=12.0, sigma_n=0.5, temps=(1.0,)),
}

CONFIG_NAMES = {
    1: "B4_k4_V1024_fp32_gauss",
    2: "B32_k5_V32000_bf16_peaks",
    3: "B64_k4_V128256_bf16_zipf_T0.7",
    4: "B256_k8_V151936_fp32_mixedT",
    5: "B1024_k4_V128256_bf16_3class",
}


@dataclass
class Case:
    """One batch of verification inputs (host numpy arrays)."""
    target: np.ndarray       # [B, k+1, V] float32, or uint16 bf16 bit patterns
    draft: np.ndarray        # [B, k, V] same dtype
    tokens: np.ndarray       # [B, k] int32
    u_accept: np.ndarray     # [B, k] float32 in [0, 1)
    u_resample: np.ndarray   # [B] float32 in [0, 1)
    temperature: np.ndarray  # [B] float32 >= 0
    dtype: str               # "f32" | "bf16"
    name: str = ""
    meta: dict = field(default_factory=dict)

    @property
    def B(self) -> int:
        return int(self.target.shape[0])

    @property
    def k(self) -> int:
        return int(self.draft.shape[1])

    @property
    def V(self) -> int:
        return int(self.target.shape[2])

    @property
    def elem_size(self) -> int:
        return 4 if self.dtype == F32 else 2

    def subset(self, idx) -> "Case":
        """The same sequences' inputs, for the given sequence indices."""
        idx = np.asarray(idx)
        return Case(np.ascontiguousarray(self.target[idx]), np.ascontiguousarray(self.draft[idx]),
                    np.ascontiguousarray(self.tokens[idx]),
                    np.ascontiguousarray(self.u_accept[idx]),
                    np.ascontiguousarray(self.u_resample[idx]),
                    np.ascontiguousarray(self.temperature[idx]), self.dtype,
                    self.name + "[subset]", dict(self.meta))


# ------------------------------------------------------------------ bf16 bits

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); returns uint16 bits.
    Inputs here are finite."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((b >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((b + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def decode(arr: np.ndarray) -> np.ndarray:
    """float32 view of a logits array (widening bf16 bits)."""
    return bf16_bits_to_f32(arr) if arr.dtype == np.uint16 else arr


# ------------------------------------------------------------- row recipes

def _normal(rng, n, sigma):
    return rng.standard_normal(n, dtype=np.float32) * np.float32(sigma)


def _peaks_row(rng, V, sigma, n_peaks, peak, exclude=None):
    row = _normal(rng, V, sigma)
    if exclude is None:
        ids = rng.choice(V, size=n_peaks, replace=False)
    else:
        mask = np.ones(V, bool)
        mask[exclude] = False
        ids = rng.choice(np.flatnonzero(mask), size=n_peaks, replace=False)
    row[ids] += np.float32(peak)
    return row, ids


def _zipf_base(V, s):
    return (-s * np.log(np.arange(1, V + 1, dtype=np.float64))).astype(np.float32)


def _zipf_row(rng, base, perm, sigma):
    row = np.empty(base.size, np.float32)
    row[perm] = base + _normal(rng, base.size, sigma)
    return row


def _zipf_target_perm(rng, V, draft_perm, top, share):
    """Target ranking: keep round(share*top) of the draft's top ids, add the rest
    from outside that set, shuffle them into ranks 1..top, and permute the
    remaining ids randomly into ranks top+1..V."""
    top_d = draft_perm[:top]
    n_keep = int(round(share * top))
    keep = rng.choice(top_d, size=n_keep, replace=False)
    mask = np.ones(V, bool)
    mask[top_d] = False
    others = rng.choice(np.flatnonzero(mask), size=top - n_keep, replace=False)
    top_t = rng.permutation(np.concatenate([keep, others]))
    rest_mask = np.ones(V, bool)
    rest_mask[top_t] = False
    rest = rng.permutation(np.flatnonzero(rest_mask))
    return np.concatenate([top_t, rest])


def _sequence_logits(p, b, rng, k, V):
    """fp32 target [k+1,V] and draft [k,V] for sequence b of recipe p."""
    t = np.empty((k + 1, V), np.float32)
    d = np.empty((k, V), np.float32)
    r = p["recipe"]
    if r == "gauss":
        for i in range(k):
            d[i] = _normal(rng, V, p["sigma_d"])
            t[i] = d[i] + _normal(rng, V, p["sigma_n"])
        t[k] = _normal(rng, V, p["sigma_d"]) + _normal(rng, V, p["sigma_n"])
    elif r == "peaks":
        for i in range(k):
            d[i], _ = _peaks_row(rng, V, p["sigma_d"], p["n_peaks"], p["peak"])
            t[i] = d[i] + _normal(rng, V, p["sigma_n"])
        fresh, _ = _peaks_row(rng, V, p["sigma_d"], p["n_peaks"], p["peak"])
        t[k] = fresh + _normal(rng, V, p["sigma_n"])
    elif r == "zipf":
        base = _zipf_base(V, p["zipf_s"])
        for i in range(k + 1):
            perm_d = rng.permutation(V)
            if i < k:
                d[i] = _zipf_row(rng, base, perm_d, p["sigma_z"])
            perm_t = _zipf_target_perm(rng, V, perm_d, p["top"], p["share"])
            t[i] = _zipf_row(rng, base, perm_t, p["sigma_z"])
    elif r == "classes":
        cls = b % 3
        for i in range(k + 1):
            drow, ids = _peaks_row(rng, V, p["sigma_d"], p["n_peaks"], p["peak"])
            if i < k:
                d[i] = drow
            if cls == 0:
                t[i] = drow  # bit-identical target (acceptance 1); fresh for the bonus row
            elif cls == 1:
                t[i], _ = _peaks_row(rng, V, p["sigma_d"], p["n_peaks"], p["peak"],
                                     exclude=ids)
            else:
                t[i] = drow + _normal(rng, V, p["sigma_n"])
    else:
        raise ValueError(f"unknown recipe {r}")
    return t, d


def _sample_tokens(rng, d_rows, T):
    """Draft tokens g_i ~ softmax(d_i / T) by Gumbel-max; argmax d_i when T == 0."""
    k, V = d_rows.shape
    g = np.empty(k, np.int32)
    for i in range(k):
        row = d_rows[i].astype(np.float64)
        if T == 0.0:
            g[i] = int(np.argmax(row))
        else:
            e = rng.standard_exponential(V)
            g[i] = int(np.argmax(row / float(T) - np.log(e)))
    return g


def make_case(params: dict, seed: int, name: str = "", threads: int | None = None) -> Case:
    """Generate one batch by a recipe dict (see CONFIGS)."""
    B, k, V, dtype = int(params["B"]), int(params["k"]), int(params["V"]), params["dtype"]
    st = np.dtype(np.float32) if dtype == F32 else np.dtype(np.uint16)
    target = np.empty((B, k + 1, V), st)
    draft = np.empty((B, k, V), st)
    tokens = np.empty((B, k), np.int32)

    urng = np.random.default_rng(seed + 2)
    u_accept = urng.random((B, k), dtype=np.float32)
    u_resample = urng.random(B, dtype=np.float32)
    temps = np.asarray(params["temps"], np.float32)
    if temps.size == 1:
        temperature = np.full(B, temps[0], np.float32)
    else:
        temperature = temps[urng.integers(0, temps.size, size=B)]

    lseeds = np.random.SeedSequence(seed).spawn(B)
    tseeds = np.random.SeedSequence(seed + 1).spawn(B)

    def one(b):
        t, d = _sequence_logits(params, b, np.random.default_rng(lseeds[b]), k, V)
        if dtype == BF16:
            target[b] = f32_to_bf16_bits(t)
            draft[b] = f32_to_bf16_bits(d)
            dd = bf16_bits_to_f32(draft[b])
        else:
            target[b] = t
            draft[b] = d
            dd = d
        tokens[b] = _sample_tokens(np.random.default_rng(tseeds[b]), dd, float(temperature[b]))

    nthr = threads or min(32, os.cpu_count() or 1)
    if nthr <= 1 or B == 1:
        for b in range(B):
            one(b)
    else:
        with ThreadPoolExecutor(nthr) as ex:
            list(ex.map(one, range(B)))
    return Case(target, draft, tokens, u_accept, u_resample, temperature, dtype,
                name or params.get("name", ""), dict(params, seed=seed))


def config_params(cfg: int, **overrides) -> dict:
    p = dict(CONFIGS[cfg])
    p.update(overrides)
    return p


def make_config(cfg: int, B: int | None = None, V: int | None = None, k: int | None = None,
                seed_offset: int = 0, threads: int | None = None) -> Case:
    """Workload `cfg` (1..5).  B/V/k overrides keep the recipe at a smaller size
    (parity tests); the full-size workload uses none."""
    over = {}
    if B is not None:
        over["B"] = B
    if V is not None:
        over["V"] = V
    if k is not None:
        over["k"] = k
    p = config_params(cfg, **over)
    name = CONFIG_NAMES[cfg] if not over else f"cfg{cfg}-recipe B{p['B']} k{p['k']} V{p['V']}"
    return make_case(p, seed=1000 * cfg + seed_offset, name=name, threads=threads)


def gauss_case(B: int, k: int, V: int, dtype: str = F32, seed: int = 7, T=1.0,
               sigma_d: float = 3.0, sigma_n: float = 0.7) -> Case:
    """Small gaussian-recipe case of any shape (edge-case tests).  T may be a
    scalar or a tuple of temperatures to draw from per sequence."""
    temps = tuple(T) if isinstance(T, (tuple, list)) else (float(T),)
    p = dict(B=B, k=k, V=V, dtype=dtype, recipe="gauss", sigma_d=sigma_d, sigma_n=sigma_n,
             temps=temps)
    return make_case(p, seed=seed, name=f"gauss B{B} k{k} V{V} {dtype}")


def algorithmic_bytes(case: Case) -> int:
    """Bytes the step must read once: all k+1 target rows of every sequence and,
    for sequences with T > 0, all k draft rows (the greedy rule never looks at
    draft logits)."""
    n_sampling = int(np.count_nonzero(case.temperature > 0))
    rows = case.B * (case.k + 1) + n_sampling * case.k
    return rows * case.V * case.elem_size


# ------------------------------------------------------------------ sampling

@dataclass
class SampleCase:
    """One batch of sampling inputs (host numpy arrays): one token per row."""
    logits: np.ndarray       # [R, V] float32, or uint16 bf16 bit patterns
    u: np.ndarray            # [R] float32 in [0, 1)
    temperature: np.ndarray  # [R] float32 >= 0
    dtype: str
    name: str = ""

    @property
    def R(self) -> int:
        return int(self.logits.shape[0])

    @property
    def V(self) -> int:
        return int(self.logits.shape[1])

    @property
    def elem_size(self) -> int:
        return 4 if self.dtype == F32 else 2


def sample_case_from(case: Case, seed: int, name: str = "") -> SampleCase:
    """The draft rows of a verification case as sampling inputs: the logits the
    draft model samples its k tokens from, each sequence's temperature for its
    k rows, and a fresh uniform per row (numpy PCG64, `seed`)."""
    R = case.B * case.k
    logits = np.ascontiguousarray(case.draft.reshape(R, case.V))
    temperature = np.repeat(case.temperature, case.k).astype(np.float32)
    u = np.random.default_rng(seed).random(R, dtype=np.float32)
    return SampleCase(logits, u, temperature, case.dtype,
                      name or f"draft rows of {case.name}")


def make_sample_config(cfg: int, B: int | None = None, V: int | None = None,
                       k: int | None = None, seed_offset: int = 0,
                       threads: int | None = None) -> SampleCase:
    """Sampling workload from workload `cfg`'s draft rows (R = B*k rows)."""
    case = make_config(cfg, B=B, V=V, k=k, seed_offset=seed_offset, threads=threads)
    name = (f"sample_R{case.B * case.k}_V{case.V}_{case.dtype}_cfg{cfg}rows"
            if B is None and V is None and k is None else "")
    return sample_case_from(case, seed=1000 * cfg + 3 + seed_offset, name=name)


def sample_bytes(sc: SampleCase) -> int:
    """Bytes a sampling call must read once: every row of every valid-T row
    (rows whose temperature is invalid are never read)."""
    T = sc.temperature
    ok = ~(np.isnan(T) | (T < 0) | np.isinf(T) | ((T > 0) & (T < np.finfo(np.float32).tiny)))
    return int(np.count_nonzero(ok)) * sc.V * sc.elem_size


# ----------------------------------------------- LM-head-fused verification

@dataclass
class LmheadCase:
    """Inputs of the LM-head-fused verification (host numpy arrays)."""
    hidden: np.ndarray       # [B, k+1, d] uint16 bf16 bits: target hidden states
    lm_head: np.ndarray      # [V, d] uint16 bf16 bits: W
    draft: np.ndarray        # [B, k, V] float32, or uint16 bf16 bits
    tokens: np.ndarray       # [B, k] int32
    u_accept: np.ndarray     # [B, k] float32
    u_resample: np.ndarray   # [B] float32
    temperature: np.ndarray  # [B] float32
    dtype: str               # the draft's dtype
    name: str = ""

    @property
    def B(self) -> int:
        return int(self.hidden.shape[0])

    @property
    def k(self) -> int:
        return int(self.hidden.shape[1]) - 1

    @property
    def d(self) -> int:
        return int(self.hidden.shape[2])

    @property
    def V(self) -> int:
        return int(self.lm_head.shape[0])


def make_lmhead_case(B: int, k: int, V: int, d: int, dtype: str = BF16, recipe: str = "grid",
                     seed: int = 11, T=(1.0,), sigma_h: float = 0.3,
                     draft_product: str = "f64") -> LmheadCase:
    """Random target hidden states and LM head, and draft logits from a draft
    model that shares the head but sees perturbed hidden states.

    recipe "grid": h in {-4..4}/4 and W in {-8..8}/32, so every product and
    partial sum of h.W is a multiple of 2^-7 below 2^17 in size: the logits
    are exact in fp32 whatever the order of accumulation (d <= 4096), and
    their spread is about sqrt(d/100).
    recipe "gauss": h ~ N(0, 1), W ~ N(0, (2.5 / sqrt d)^2), both rounded to
    bf16: logits of spread about 2.5, rounded by any fp32 accumulation.
    Draft hidden states are the target's plus N(0, sigma_h^2) per element
    (on the grid recipe rounded back to the grid); draft logits are their
    product with W in float64 (draft_product="f32": in float32, for the
    full-size shapes), stored as `dtype`.  Draft tokens are sampled
    from the draft logits at the sequence's temperature (argmax at T = 0);
    uniforms are float32 in [0, 1).  The bonus position has no draft row."""
    rng = np.random.default_rng(seed)
    if recipe == "grid":
        h = rng.integers(-4, 5, size=(B, k + 1, d)).astype(np.float32) / 4.0
        w = rng.integers(-8, 9, size=(V, d)).astype(np.float32) / 32.0
        hd = h[:, :k] + np.round(rng.normal(0.0, sigma_h, size=(B, k, d)) * 4.0) / 4.0
        hd = np.clip(hd, -1.0, 1.0).astype(np.float32)
    elif recipe == "gauss":
        h = rng.standard_normal((B, k + 1, d), dtype=np.float32)
        w = rng.standard_normal((V, d), dtype=np.float32) * np.float32(2.5 / np.sqrt(d))
        hd = h[:, :k] + rng.standard_normal((B, k, d), dtype=np.float32) * np.float32(sigma_h)
    else:
        raise ValueError(f"unknown recipe {recipe}")
    hb = f32_to_bf16_bits(h)
    wb = f32_to_bf16_bits(w)
    hdb = f32_to_bf16_bits(hd)
    if draft_product == "f32":
        dl32 = (bf16_bits_to_f32(hdb).reshape(-1, d) @ bf16_bits_to_f32(wb).T).reshape(B, k, V)
    else:
        w64 = bf16_bits_to_f32(wb).astype(np.float64)
        dl = (bf16_bits_to_f32(hdb).astype(np.float64).reshape(-1, d) @ w64.T).reshape(B, k, V)
        dl32 = dl.astype(np.float32)
    draft = f32_to_bf16_bits(dl32) if dtype == BF16 else dl32
    temps = tuple(T) if isinstance(T, (tuple, list)) else (float(T),)
    temperature = np.asarray(rng.choice(temps, size=B), np.float32)
    rows = decode(draft)
    tokens = np.stack([_sample_tokens(rng, rows[b], float(temperature[b])) for b in range(B)])
    u_accept = rng.random((B, k), dtype=np.float32)
    u_resample = rng.random(B, dtype=np.float32)
    return LmheadCase(hb, wb, draft, tokens.astype(np.int32), u_accept, u_resample,
                      temperature, dtype, name=f"lmhead {recipe} B{B} k{k} V{V} d{d} {dtype}")


def lmhead_flops(c: LmheadCase) -> int:
    """Multiply-add flops of the statistics GEMM (2 per product, B(k+1) rows)."""
    return 2 * c.B * (c.k + 1) * c.V * c.d


# ------------------------------------------------------- tree verification

@dataclass
class TreeCase:
    """One batch of tree-verification inputs (host numpy arrays).  Node 0 is
    the root; node n >= 1 holds tokens[b, n] below parent[b, n] < n."""
    target: np.ndarray       # [B, N, V] float32, or uint16 bf16 bit patterns
    draft: np.ndarray        # [B, N, V] same dtype
    parent: np.ndarray       # [B, N] int32 (entry 0: -1)
    tokens: np.ndarray       # [B, N] int32 (entry 0: -1)
    n_nodes: np.ndarray      # [B] int32
    u_accept: np.ndarray     # [B, N] float32 in [0, 1)
    u_resample: np.ndarray   # [B] float32 in [0, 1)
    temperature: np.ndarray  # [B] float32 >= 0
    dtype: str
    name: str = ""
    meta: dict = field(default_factory=dict)

    @property
    def B(self) -> int:
        return int(self.target.shape[0])

    @property
    def N(self) -> int:
        return int(self.target.shape[1])

    @property
    def V(self) -> int:
        return int(self.target.shape[2])

    @property
    def elem_size(self) -> int:
        return 4 if self.dtype == F32 else 2

    def subset(self, idx) -> "TreeCase":
        idx = np.asarray(idx)
        c = lambda a: np.ascontiguousarray(a[idx])
        return TreeCase(c(self.target), c(self.draft), c(self.parent), c(self.tokens),
                        c(self.n_nodes), c(self.u_accept), c(self.u_resample),
                        c(self.temperature), self.dtype, self.name + "[subset]",
                        dict(self.meta))


def tree_shape(branching) -> np.ndarray:
    """Parent array of the full tree whose depth-l nodes each have
    branching[l] children, nodes numbered breadth first (root 0, parent[0] =
    -1)."""
    parent = [-1]
    level = [0]
    for w in branching:
        nxt = []
        for c in level:
            for _ in range(int(w)):
                parent.append(c)
                nxt.append(len(parent) - 1)
        level = nxt
    return np.asarray(parent, np.int32)


TREE_CONFIGS = {
    # small: the oracle finishes in well under a second
    1: dict(B=8, V=1024, dtype=F32, branching=(2, 2, 1), recipe="gauss", sigma_d=3.0,
            sigma_n=0.7, temps=(0.0, 1.0), ragged=True),
    # full size: a 29-node tree (4 first-level candidates, 2 below each, two
    # more levels of single continuations) over a 128256-token vocabulary
    2: dict(B=512, V=128256, dtype=BF16, branching=(4, 2, 1, 1), recipe="gauss",
            sigma_d=2.0, sigma_n=0.5, temps=(0.0, 0.7, 1.0), ragged=False),
}

TREE_CONFIG_NAMES = {
    1: "tree_B8_N11_V1024_fp32",
    2: "tree_B512_N29_V128256_bf16",
}


def _tree_children_tokens(rng, drow, m, T):
    """m children of a node: independent Gumbel-max draws from softmax(d/T),
    or the m largest draft logits (distinct, descending; repeated cyclically
    when m exceeds the vocabulary) when T == 0."""
    if m == 0:
        return np.empty(0, np.int32)
    row = drow.astype(np.float64)
    if T == 0.0:
        order = np.lexsort((np.arange(row.size), -row))
        return order[np.arange(m) % row.size].astype(np.int32)
    out = np.empty(m, np.int32)
    for i in range(m):
        e = rng.standard_exponential(row.size)
        out[i] = int(np.argmax(row / float(T) - np.log(e)))
    return out


def make_tree_case(params: dict, seed: int, name: str = "",
                   threads: int | None = None) -> TreeCase:
    """Generate one batch of trees.  Every node's draft row follows the recipe
    (gauss: N(0, sigma_d^2); peaks: as workload 2) and its target row is the
    draft row plus N(0, sigma_n^2).  Children are drawn from their parent's
    draft row (_tree_children_tokens).  With ragged=True each sequence keeps a
    random breadth-first prefix of the tree (n_nodes in [1, N]), the rest
    padded with parent/token -1 and zero rows."""
    B, V, dtype = int(params["B"]), int(params["V"]), params["dtype"]
    shape = tree_shape(params["branching"])
    N = int(shape.size)
    st = np.dtype(np.float32) if dtype == F32 else np.dtype(np.uint16)
    target = np.zeros((B, N, V), st)
    draft = np.zeros((B, N, V), st)
    parent = np.tile(shape, (B, 1))
    tokens = np.full((B, N), -1, np.int32)

    urng = np.random.default_rng(seed + 2)
    u_accept = urng.random((B, N), dtype=np.float32)
    u_resample = urng.random(B, dtype=np.float32)
    temps = np.asarray(params["temps"], np.float32)
    temperature = temps[urng.integers(0, temps.size, size=B)]
    if params.get("ragged"):
        n_nodes = urng.integers(1, N + 1, size=B).astype(np.int32)
        n_nodes[0] = N
    else:
        n_nodes = np.full(B, N, np.int32)

    lseeds = np.random.SeedSequence(seed).spawn(B)
    tseeds = np.random.SeedSequence(seed + 1).spawn(B)

    def one(b):
        rng = np.random.default_rng(lseeds[b])
        trng = np.random.default_rng(tseeds[b])
        n = int(n_nodes[b])
        T = float(temperature[b])
        for c in range(n):
            if params["recipe"] == "peaks":
                d, _ = _peaks_row(rng, V, params["sigma_d"], params["n_peaks"], params["peak"])
            else:
                d = _normal(rng, V, params["sigma_d"])
            t = d + _normal(rng, V, params["sigma_n"])
            if dtype == BF16:
                draft[b, c] = f32_to_bf16_bits(d)
                target[b, c] = f32_to_bf16_bits(t)
                dd = bf16_bits_to_f32(draft[b, c])
            else:
                draft[b, c] = d
                target[b, c] = t
                dd = d
            kids = [i for i in range(c + 1, n) if shape[i] == c]
            tokens[b, kids] = _tree_children_tokens(trng, dd, len(kids), T)
        parent[b, n:] = -1

    nthr = threads or min(32, os.cpu_count() or 1)
    if nthr <= 1 or B == 1:
        for b in range(B):
            one(b)
    else:
        with ThreadPoolExecutor(nthr) as ex:
            list(ex.map(one, range(B)))
    return TreeCase(target, draft, parent, tokens, n_nodes, u_accept, u_resample, temperature,
                    dtype, name or params.get("name", ""), dict(params, seed=seed))


def make_tree_config(cfg: int, B: int | None = None, V: int | None = None,
                     seed_offset: int = 0, threads: int | None = None) -> TreeCase:
    """Tree workload `cfg` (TREE_CONFIGS); B/V overrides keep the recipe."""
    p = dict(TREE_CONFIGS[cfg])
    if B is not None:
        p["B"] = B
    if V is not None:
        p["V"] = V
    name = TREE_CONFIG_NAMES[cfg] if B is None and V is None else \
        f"tree{cfg}-recipe B{p['B']} V{p['V']}"
    return make_tree_case(p, seed=5000 + 1000 * cfg + seed_offset, name=name, threads=threads)


def tree_bytes(tc: TreeCase, out_nodes: np.ndarray, num_accepted: np.ndarray) -> int:
    """Bytes a tree verification must read once, given the walk's result:
    the target row of every visited node (the root and the accepted path)
    and, at T > 0, the draft row of every visited node that has children."""
    rows = 0
    for b in range(tc.B):
        na = int(num_accepted[b])
        if na < 0:
            continue
        visited = [0] + [int(x) for x in out_nodes[b, :na]]
        n = int(tc.n_nodes[b])
        par = tc.parent[b, :n]
        for c in visited:
            rows += 1
            if tc.temperature[b] > 0 and np.any(par[c + 1:] == c):
                rows += 1
    return rows * tc.V * tc.elem_size
