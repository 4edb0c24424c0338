"""A seeded random sweep of tree topologies for the Medusa walk and for recursive rejection
(children i.i.d. and without replacement) against the fp64 oracle.

Random recursive trees (each node's parent drawn from the root and the nodes before it, at
most a dozen children per node), batch sizes, vocabularies (16-byte rows and not), dtypes,
drafter noise and temperature mixes come from one seeded generator; the comparisons are
those of tests/test_gpu_tree.py and tests/test_gpu_tree_rr.py (exact, except draws flagged
at a decision or CDF boundary)."""
import numpy as np
import pytest
import torch

import workloads
from test_gpu_tree import _check_tree
from test_gpu_tree_rr import KEYS, Report, check_walks

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def sd(built_library):
    import speculative_decoding_token_temperature_gb300 as m
    m.load_library()
    return m


def _topology(rng, N, max_kids):
    parents, kids, depth = [], {-1: 0}, {-1: 0}
    for i in range(N):
        while True:
            a = int(rng.integers(-1, i))
            if kids.get(a, 0) < max_kids:
                break
        parents.append(a)
        kids[a] = kids.get(a, 0) + 1
        depth[i] = depth[a] + 1
    return parents, max(depth.values())


def _cases(seed, n):
    rng = np.random.default_rng(seed)
    for _ in range(n):
        V = int([rng.integers(8, 200), rng.integers(200, 5000), rng.integers(5000, 40000)][rng.integers(0, 3)])
        if rng.random() < 0.6:
            V -= V % 8
        N = int(rng.integers(1, 160))
        parents, D = _topology(rng, N, min(12, V))
        yield dict(V=V, N=N, parents=parents, D=D, B=int(rng.integers(1, 17)),
                   dtype=["bf16", "fp32"][rng.integers(0, 2)], noise=float(rng.choice([0.3, 1.0, 2.0])),
                   temps=str(rng.choice(["const:1.0", "uniform:0.0:1.5", "half_greedy:0.7"])),
                   seed=int(rng.integers(0, 2**31)))


def _inputs(c, wor):
    return workloads.make_tree_rr_inputs(c["B"], c["V"], c["parents"], depth=c["D"], seed=c["seed"], device=DEV,
                                         dtype=c["dtype"], scale=2.0, n_spikes=min(8, c["V"]), spike=4.0,
                                         noise=c["noise"], temps=c["temps"], without_replacement=wor)


@pytest.mark.parametrize("wor", [False, True])
def test_random_trees_recursive_rejection(sd, wor):
    rep = Report(f"random trees, recursive rejection, without replacement={wor}")
    for i, c in enumerate(_cases(21 + int(wor), 12)):
        x = _inputs(c, wor)
        out = sd.verify_tree_recursive(*(x[k] for k in KEYS), c["D"], without_replacement=wor)
        torch.cuda.synchronize()
        n0 = len(rep.failures)
        check_walks(rep, x, out, c["D"], wor=wor)
        assert len(rep.failures) == n0, (i, {k: c[k] for k in ("V", "N", "D", "B", "dtype")}, rep.failures[n0:n0 + 3])
    rep.finish(budget=False)


def test_random_trees_medusa_walk(sd):
    stats = {"sequences": 0, "flagged": 0, "accepted": 0}
    for c in _cases(23, 12):
        x = _inputs(c, False)
        D = c["D"]
        out = sd.verify_tree(x["logits"], x["node_tokens"], x["parents"], x["temperatures"],
                             x["uniforms"][:, :D + 1].contiguous(), D)
        torch.cuda.synchronize()
        y = dict(x)
        y["uniforms"] = x["uniforms"][:, :D + 1].contiguous()
        _check_tree(out, y, D, stats)
    assert stats["sequences"] > 0
