"""GPU parity of the Medusa tree walk and the tree-attention mask (via the C ABI)."""
import json
import os

import numpy as np
import pytest
import torch

import workloads
from golden import read_fixture
from oracle import specdec_oracle as so
from parity import FLAG_TOL, assert_flag_budget

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def sd(built_library):
    import speculative_decoding_token_temperature_gb300 as m
    m.load_library()
    return m


@pytest.fixture(scope="module")
def medusa64():
    parents, paths, _ = so.medusa_sparse_tree(workloads.medusa_workload_accuracies(), 64)
    return parents, paths


def _np(t):
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.detach().cpu().numpy()


def _check_tree(gpu, x, D, stats):
    L, toks, par = _np(x["logits"]), _np(x["node_tokens"]), _np(x["parents"])
    T, u = _np(x["temperatures"]), _np(x["uniforms"])
    B = L.shape[0]
    for b in range(B):
        o = so.verify_tree_sequence(L[b], toks[b], par, float(T[b]), u[b], D)
        gt, gp, gJ, gs = (_np(gpu[k])[b] for k in ("tokens", "path", "num_accepted", "status"))
        gJ, gs = int(gJ), int(gs)
        stats["sequences"] += 1
        assert gs == o["status"], (b, gs, o["status"])
        if o["status"] & 0xFF:
            assert gJ == -1 and (gt == -1).all() and (gp == -1).all()
            continue
        if np.array_equal(gt, o["tokens"]) and np.array_equal(gp, o["path"]) and gJ == o["n_accepted"]:
            stats["accepted"] += gJ
            continue
        # the walks may differ only at a flagged draw: first differing depth
        assert float(T[b]) >= so.GREEDY_T, f"greedy walk differs at seq {b}: {gt} vs {o['tokens']}"
        d = int(np.flatnonzero(gt != o["tokens"])[0])
        node = -1 if d == 0 else int(o["path"][d - 1])
        row = L[b][0 if node < 0 else 1 + node]
        p = so.target_distribution(row, float(T[b]))
        _, C, S = so.inverse_cdf(p, u[b][d])
        y = int(gt[d])
        lo = (C[y - 1] if y > 0 else 0.0) / S
        hi = C[y] / S
        assert p[y] > 0 and lo - FLAG_TOL <= u[b][d] <= hi + FLAG_TOL, (b, d, y, lo, hi, u[b][d])
        stats["flagged"] += 1


def test_tree_b32_n64_v32000(sd, medusa64):
    parents, paths = medusa64
    stats = {"sequences": 0, "flagged": 0, "accepted": 0}
    for r in range(100):
        x = workloads.tree_workload("tree_b32_n64_v32000", parents, paths, r, DEV)
        out = sd.verify_tree(x["logits"], x["node_tokens"], x["parents"], x["temperatures"], x["uniforms"], 4)
        torch.cuda.synchronize()
        _check_tree(out, x, 4, stats)
    path = os.environ.get("SPECDEC_PARITY_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"workload": "tree_b32_n64_v32000 (100 rounds)", **stats}) + "\n")
    assert_flag_budget(stats["flagged"], stats["sequences"] * 5, stats)  # up to D + 1 = 5 draws a walk
    assert stats["accepted"] > 0


@pytest.mark.parametrize("C", ["1", "2", "4", "8"])
@pytest.mark.parametrize("V,dtype", [(32008, "bf16"), (20004, "fp32"), (64, "bf16")])
def test_tree_cluster_sizes(sd, medusa64, hooks, C, V, dtype):
    """Rows split across clusters of 1, 2, 4 and 8 CTAs (a short last slice at V = 32008
    and 20004; at V = 64 each CTA of an 8-CTA cluster holds a single 16-byte vector).
    Spiked logits (1 N(0,1), +10 on child tokens) make most walks descend several levels."""
    parents, paths = medusa64
    hooks(tree_cluster=int(C))
    stats = {"sequences": 0, "flagged": 0, "accepted": 0}
    for seed in range(3):
        x = workloads.make_tree_inputs(12, V, parents, paths, depth=4, seed=100 * seed + V % 97, device=DEV,
                                       dtype=dtype, top=min(10, V), scale=1.0, spike=10.0,
                                       temps="half_greedy:0.7")
        out = sd.verify_tree(x["logits"], x["node_tokens"], x["parents"], x["temperatures"], x["uniforms"], 4)
        _check_tree(out, x, 4, stats)
    assert stats["accepted"] >= stats["sequences"]  # walks descend on average at least once
    assert stats["flagged"] <= 1


def test_tree_v128256_rows_split(sd, medusa64):
    """A 128256-entry vocabulary (256 KB bf16 rows, staged as four 64 KB slices)."""
    parents, paths = medusa64
    stats = {"sequences": 0, "flagged": 0, "accepted": 0}
    x = workloads.make_tree_inputs(16, 128256, parents, paths, depth=4, seed=9, device=DEV, dtype="bf16",
                                   scale=1.0, spike=12.0, temps="half_greedy:0.9")
    out = sd.verify_tree(x["logits"], x["node_tokens"], x["parents"], x["temperatures"], x["uniforms"], 4)
    _check_tree(out, x, 4, stats)
    assert stats["accepted"] > 0 and stats["flagged"] <= 1


def test_tree_large_tree_block_child_search(sd):
    """A 4680-node tree (4 heads x top-8, every path): more nodes than one warp searches, so
    the cluster walk finds children with the whole CTA; spiked logits make walks descend."""
    from fractions import Fraction
    acc = [[Fraction(1, 2 + i + k).limit_denominator(1000) for i in range(8)] for k in range(4)]
    parents, paths, _ = so.medusa_sparse_tree(acc, 10 ** 6)
    assert len(parents) == 4680
    stats = {"sequences": 0, "flagged": 0, "accepted": 0}
    for seed, dtype in ((1, "bf16"), (2, "fp32")):
        x = workloads.make_tree_inputs(4, 2048, parents, paths, depth=4, seed=seed, device=DEV, dtype=dtype,
                                       top=8, scale=1.0, spike=10.0)
        out = sd.verify_tree(x["logits"], x["node_tokens"], x["parents"], x["temperatures"], x["uniforms"], 4)
        _check_tree(out, x, 4, stats)
    assert stats["accepted"] >= stats["sequences"]
    assert stats["flagged"] <= 1


def test_tree_deep_walks_b32(sd, medusa64):
    """tree_b32_n64_v32000's shapes with logits whose spikes dominate, so walks reach the
    deepest levels (the stated workload's spikes rarely win, and its walks stop at the root)."""
    parents, paths = medusa64
    stats = {"sequences": 0, "flagged": 0, "accepted": 0}
    for r in range(6):
        x = workloads.make_tree_inputs(32, 32000, parents, paths, depth=4, seed=500 + r, device=DEV,
                                       scale=1.0, spike=10.0)
        out = sd.verify_tree(x["logits"], x["node_tokens"], x["parents"], x["temperatures"], x["uniforms"], 4)
        _check_tree(out, x, 4, stats)
    assert stats["accepted"] >= 1.5 * stats["sequences"]
    assert stats["flagged"] <= 1


@pytest.mark.parametrize("V,dtype", [(32000, "bf16"), (1001, "fp32"), (4096, "fp32"), (37, "bf16")])
def test_tree_shapes_and_edges(sd, medusa64, V, dtype):
    parents, paths = medusa64
    stats = {"sequences": 0, "flagged": 0, "accepted": 0}
    x = workloads.make_tree_inputs(8, V, parents, paths, depth=4, seed=V, device=DEV, dtype=dtype,
                                   top=min(10, V))
    out = sd.verify_tree(x["logits"], x["node_tokens"], x["parents"], x["temperatures"], x["uniforms"], 4)
    _check_tree(out, x, 4, stats)


def test_tree_degenerate(sd):
    V, D = 50, 3
    parents = torch.tensor([-1, -1, 0, 0, 2], dtype=torch.int32, device=DEV)
    B = 6
    g = torch.Generator(device=DEV).manual_seed(2)
    logits = torch.randn(B, 6, V, generator=g, device=DEV)
    toks = torch.randint(0, V, (B, 5), generator=g, device=DEV, dtype=torch.int32)
    toks[0, 0] = toks[0, 1] = int(torch.argmax(logits[0, 0]))      # duplicate siblings
    toks[1, 3] = V + 1                                               # bad token
    logits[2, 0, 4] = float("nan")                                   # bad root row
    T = torch.tensor([0.0, 0.5, 0.5, 0.5, 0.0, 0.9], device=DEV)
    u = torch.rand(B, D + 1, generator=g, device=DEV)
    u[3, 2] = 1.5                                                    # bad uniform
    out = sd.verify_tree(logits, toks, parents, T, u, D)
    x = {"logits": logits, "node_tokens": toks, "parents": parents, "temperatures": T, "uniforms": u}
    _check_tree(out, x, D, {"sequences": 0, "flagged": 0, "accepted": 0})
    # too deep for max_depth 2, and a bad parent
    out = sd.verify_tree(logits, toks, parents, T, u[:, :3].contiguous(), 2)
    assert (out["status"].cpu() & so.STATUS_BAD_TREE).all()
    bad = torch.tensor([-1, 1, 0, 0, 2], dtype=torch.int32, device=DEV)
    out = sd.verify_tree(logits, toks, bad, T, u, D)
    assert (out["status"].cpu() & so.STATUS_BAD_TREE).all()
    # a tree with no nodes: the root draw alone
    out = sd.verify_tree(logits[:, :1].contiguous(), toks[:, :0].contiguous(),
                         parents[:0].contiguous(), T, u, D)
    assert (out["num_accepted"].cpu()[[0, 1, 4, 5]] == 0).all()


@pytest.mark.parametrize("C", ["1", "4"])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_tree_degenerate_cluster_walk(sd, hooks, C, dtype):
    """The input errors of test_tree_degenerate on 16-byte rows (the cluster walk), plus
    errors in rows the walk reaches only after descending, and in rows it never reads."""
    hooks(tree_cluster=int(C))
    V, D = 1024, 3
    parents = torch.tensor([-1, -1, 0, 0, 2], dtype=torch.int32, device=DEV)
    B = 10
    g = torch.Generator(device=DEV).manual_seed(3)
    logits = torch.randn(B, 6, V, generator=g, device=DEV)
    toks = torch.randint(0, V, (B, 5), generator=g, device=DEV, dtype=torch.int32)
    for b in range(B):  # spike the first child's token in every row, so walks descend
        for row, node in ((0, 0), (1, 2), (3, 4)):
            logits[b, row, int(toks[b, node])] += 12.0
    toks[0, 0] = toks[0, 1] = int(torch.argmax(logits[0, 0]))      # duplicate siblings
    toks[1, 3] = V + 1                                               # bad token
    logits[2, 0, 4] = float("nan")                                   # bad root row
    logits[5, 1, 7] = float("nan")                                   # bad row of node 0 (reached by descent)
    logits[6, 2, :] = float("-inf")                                  # node 1's row: never reached
    logits[7, 1, :] = float("-inf")                                  # node 0's row empty
    logits[8, 5, 9] = float("inf")                                   # a leaf's row: never read
    T = torch.tensor([0.0, 0.5, 0.5, 0.5, 0.0, 0.9, 0.7, 0.0, 0.6, float("nan")], device=DEV)
    u = torch.rand(B, D + 1, generator=g, device=DEV)
    u[3, 2] = 1.5                                                    # bad uniform
    if dtype == "bf16":
        logits = logits.to(torch.bfloat16)
    out = sd.verify_tree(logits, toks, parents, T, u, D)
    x = {"logits": logits, "node_tokens": toks, "parents": parents, "temperatures": T, "uniforms": u}
    _check_tree(out, x, D, {"sequences": 0, "flagged": 0, "accepted": 0})
    out = sd.verify_tree(logits, toks, parents, T, u[:, :3].contiguous(), 2)  # too deep for max_depth 2
    assert (out["status"].cpu() & so.STATUS_BAD_TREE).all()
    bad = torch.tensor([-1, 1, 0, 0, 2], dtype=torch.int32, device=DEV)
    out = sd.verify_tree(logits, toks, bad, T, u, D)
    assert (out["status"].cpu() & so.STATUS_BAD_TREE).all()


def test_mask_worked_example(sd):
    fx = read_fixture("tree_mask_6node.txt")
    parents = torch.tensor([int(v) for v in fx["parents"]], dtype=torch.int32, device=DEV)
    P = 3
    r = sd.build_tree_mask(parents, P)
    block = np.array([[int(v) for v in row] for row in fx["mask_row"]], dtype=np.uint8)
    m = _np(r["mask"])
    assert (m[:, :P] == 1).all()
    assert np.array_equal(m[:, P:], block)
    assert _np(r["depth"]).tolist() == [int(v) for v in fx["depth"]]
    assert _np(r["position_ids"]).tolist() == [P + int(v) for v in fx["depth"]]
    assert int(r["status"][0]) == 0


@pytest.mark.parametrize("which", ["medusa64", "full4680", "chain", "random"])
def test_mask_matches_oracle(sd, which):
    if which == "medusa64":
        parents, _, _ = so.medusa_sparse_tree(workloads.medusa_workload_accuracies(), 64)
    elif which == "full4680":
        acc = [[1 / (2 + i + k) for i in range(8)] for k in range(4)]
        from fractions import Fraction
        acc = [[Fraction(a).limit_denominator(1000) for a in h] for h in acc]
        parents, _, _ = so.medusa_sparse_tree(acc, 10 ** 6)
        assert len(parents) == 4680
    elif which == "chain":
        parents = list(range(-1, 99))
    else:
        rng = np.random.default_rng(4)
        parents = [-1] + [int(rng.integers(-1, i)) for i in range(1, 300)]
    P = 17
    r = sd.build_tree_mask(torch.tensor(parents, dtype=torch.int32, device=DEV), P)
    mask, pos, depth = so.build_tree_mask(parents, P)
    assert np.array_equal(_np(r["mask"]).astype(bool), mask)
    assert np.array_equal(_np(r["position_ids"]), pos)
    assert np.array_equal(_np(r["depth"]), depth)


def test_mask_bad_parents(sd):
    r = sd.build_tree_mask(torch.tensor([-1, 0, 5, 1], dtype=torch.int32, device=DEV), 2)
    assert int(r["status"][0]) == so.STATUS_BAD_TREE


@pytest.mark.parametrize("P", [0, 1, 15, 16, 33, 100])
@pytest.mark.parametrize("offset", [0, 1, 7])
def test_mask_rows_of_every_alignment(sd, P, offset):
    """Rows of P + N bytes start at every offset modulo 16, and the mask itself may start
    off a 16-byte boundary (a byte offset into a larger buffer, through the C ABI): the
    kernel's word stores and byte ends must give the oracle's mask exactly."""
    import ctypes
    rng = np.random.default_rng(P * 10 + offset)
    lib = sd.load_library()
    for N in (1, 2, 5, 37, 130):
        parents = [-1] + [int(rng.integers(-1, i)) for i in range(1, N)]
        par = torch.tensor(parents, dtype=torch.int32, device=DEV)
        W = P + N
        buf = torch.full((offset + W * N + 64,), 7, dtype=torch.uint8, device=DEV)
        pos = torch.empty(N, dtype=torch.int64, device=DEV)
        dep = torch.empty(N, dtype=torch.int32, device=DEV)
        st = torch.empty(1, dtype=torch.int32, device=DEV)
        p = ctypes.c_void_p
        rc = lib.specdec_build_tree_mask(p(par.data_ptr()), N, P, p(buf.data_ptr() + offset), p(pos.data_ptr()),
                                         p(dep.data_ptr()), p(st.data_ptr()), p(torch.cuda.current_stream().cuda_stream))
        assert rc == 0
        torch.cuda.synchronize()
        mask, opos, odep = so.build_tree_mask(parents, P)
        got = _np(buf)
        assert (got[:offset] == 7).all() and (got[offset + W * N:] == 7).all(), (N, "writes outside the mask")
        assert np.array_equal(got[offset:offset + W * N].reshape(N, W).astype(bool), mask), (N, P, offset)
        assert set(np.unique(got[offset:offset + W * N])) <= {0, 1}
        assert np.array_equal(_np(pos), opos) and np.array_equal(_np(dep), odep) and int(st[0]) == 0
