"""GPU parity of sampled tree verification by recursive rejection against the fp64 oracle
(SD 20.5, box "Recursive rejection at a node with several children"), through the C ABI,
with children drafted i.i.d. and, as Sequoia does, drawn without replacement.

Rules (those of tests/parity.py, applied to a walk):
* status error bits, greedy walks (tokens, path, count): bit-exact; an error sequence has
  count -1 and -1 outputs;
* sampled walks: the same path and final token, except a FLAGGED difference: where the two
  paths first part, the first child whose decision differs must lie within FLAG_TOL of its
  boundary R(s)/q(s) in the oracle; with equal paths, a different final token must have
  positive weight with u[0] within FLAG_TOL of its interval of the oracle's CDF.  Warning
  bits are compared where the paths agree.  Flags stay within 1e-4 of the decisions
  checked (up to D + 1 per walk), with no floor.
"""
import json
import os

import numpy as np
import pytest
import torch

import workloads
from parity import FLAG_TOL, assert_flag_budget

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
KEYS = ("logits", "draft_probs", "node_tokens", "parents", "temperatures", "uniforms")


@pytest.fixture(scope="module")
def sd(built_library):
    import speculative_decoding_token_temperature_gb300 as m
    m.load_library()
    return m


@pytest.fixture(scope="module")
def medusa_parents():
    from oracle import specdec_oracle as so
    parents, _, _ = so.medusa_sparse_tree(workloads.medusa_workload_accuracies(), 64)
    return parents


def _np(t):
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.detach().cpu().numpy()


class Report:
    def __init__(self, name):
        self.name, self.sequences, self.flagged, self.nodes, self.failures = name, 0, 0, 0, []
        self.decisions = 0  # up to D + 1 per walk

    def fail(self, msg):
        if len(self.failures) < 20:
            self.failures.append(msg)

    def finish(self, budget=True):
        path = os.environ.get("SPECDEC_PARITY_REPORT")
        if path:
            with open(path, "a") as f:
                f.write(json.dumps({"workload": self.name, "rule": "tree_recursive", "sequences": self.sequences,
                                    "accepted_nodes": self.nodes, "flagged": self.flagged,
                                    "hard_failures": len(self.failures)}) + "\n")
        assert not self.failures, self.failures[:10]
        if budget:
            assert_flag_budget(self.flagged, self.decisions, self.name)


def check_walks(rep, x, out, D, wor=False):
    from oracle import specdec_oracle as so
    L, q, toks, parents, T, u = (_np(x[k]) for k in KEYS)
    g_t, g_p, g_J, g_s = (_np(out[k]) for k in ("tokens", "path", "num_accepted", "status"))
    B = L.shape[0]
    for b in range(B):
        o = so.verify_tree_rr_sequence(L[b], q[b], toks[b], parents, float(T[b]), u[b], D, want_cdf=True,
                                       without_replacement=wor)
        rep.sequences += 1
        rep.decisions += D + 1
        gs, os_ = int(g_s[b]), int(o["status"])
        if (gs & 0xFF) != (os_ & 0xFF):
            rep.fail(f"seq {b}: status gpu {gs} oracle {os_}")
            continue
        if os_ & 0xFF:
            if g_J[b] != -1 or (g_t[b] != -1).any() or (g_p[b] != -1).any():
                rep.fail(f"seq {b}: error sequence has outputs")
            continue
        rep.nodes += max(o["n_accepted"], 0)
        same_path = np.array_equal(g_p[b], o["path"]) and g_J[b] == o["n_accepted"]
        if o["greedy"]:
            if not (same_path and np.array_equal(g_t[b], o["tokens"]) and gs == os_):
                rep.fail(f"seq {b}: greedy walk differs gpu {g_t[b]} {g_p[b]} oracle {o['tokens']} {o['path']}")
            continue
        if not same_path:
            i = 0
            while i < D and g_p[b][i] == o["path"][i] and g_p[b][i] >= 0:
                i += 1
            gj = int(g_p[b][i]) if i < D and g_p[b][i] >= 0 else None
            oj = int(o["path"][i]) if i < D and o["path"][i] >= 0 else None
            first = min(j for j in (gj, oj) if j is not None) if (gj is not None or oj is not None) else None
            if first is not None and o["margins"][first] < FLAG_TOL:
                rep.flagged += 1
            else:
                rep.fail(f"seq {b}: paths part at depth {i}: gpu {g_p[b]} oracle {o['path']}")
            continue
        if (gs & 256) != (os_ & 256):
            rep.fail(f"seq {b}: ZERO_Q differs with equal paths")
            continue
        J = int(g_J[b])
        if not np.array_equal(g_t[b][:J], o["tokens"][:J]) or (g_t[b][J + 1:] != -1).any():
            rep.fail(f"seq {b}: accepted tokens or padding differ {g_t[b]} vs {o['tokens']}")
            continue
        gy, oy = int(g_t[b][J]), int(o["tokens"][J])
        if gy != oy:
            if (gs & 512) != (os_ & 512):
                rep.flagged += 1  # a zero residual decided by rounding
                continue
            C, S = o["cdf"], o["S"]
            if 0 <= gy < len(C):
                lo = (C[gy - 1] if gy > 0 else 0.0) / S
                hi = C[gy] / S
                uu = float(u[b][0])
                if hi > lo and lo - FLAG_TOL <= uu <= hi + FLAG_TOL:
                    rep.flagged += 1
                    continue
            rep.fail(f"seq {b}: final token gpu {gy} oracle {oy}")


def _run(sd, x, D, wor=False):
    out = sd.verify_tree_recursive(*(x[k] for k in KEYS), D, without_replacement=wor)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("wor", [False, True])
def test_tree_rr_medusa_topology_rounds(sd, medusa_parents, wor):
    rep = Report("tree_rr_b32_n64_v32000 (20 rounds)" + (", without replacement" if wor else ""))
    for r in range(20):
        x = workloads.tree_rr_workload("tree_rr_b32_n64_v32000", medusa_parents, r, DEV, without_replacement=wor)
        check_walks(rep, x, _run(sd, x, 4, wor), 4, wor)
    rep.finish()
    assert rep.nodes > 0


@pytest.mark.parametrize("parents,V,dtype", [
    ([-1, -1, -1, -1], 64, "bf16"),                      # one node, four children
    ([-1, 0, 1, 2, 3], 4099, "fp32"),                    # a chain (odd V: scalar loads)
    ([-1, -1, 0, 0, 1, 2, 2, 5], 50000, "bf16"),
    ([-1, -1, -1, 0, 0, 0, 1, 1, 2, 3, 3, 6], 7, "fp32"),  # 3 children of V = 7 tokens: mass used up
    ([-1] * 8, 8, "bf16"),                                # every token of V = 8 a child
])
def test_tree_rr_without_replacement_shapes(sd, parents, V, dtype):
    from oracle import specdec_oracle as so
    D = max(1, int(so.tree_depths(parents).max()) + 1)
    rep = Report(f"tree_rr without replacement N={len(parents)} V={V} {dtype}")
    for seed in range(4):
        x = workloads.make_tree_rr_inputs(6, V, parents, depth=D, seed=seed, device=DEV, dtype=dtype,
                                          scale=2.0, n_spikes=min(3, V), spike=3.0, noise=0.6,
                                          temps="uniform:0.0:1.5", without_replacement=True)
        check_walks(rep, x, _run(sd, x, D, True), D, True)
    rep.finish(budget=False)


@pytest.mark.parametrize("C", ["1", "2", "4", "8"])
def test_tree_rr_without_replacement_cluster_sizes(sd, medusa_parents, hooks, C):
    hooks(tree_cluster=int(C))
    rep = Report(f"tree_rr without replacement cluster {C}")
    for seed in range(3):
        x = workloads.make_tree_rr_inputs(8, 32008, medusa_parents, depth=4, seed=60 + seed, device=DEV,
                                          dtype="bf16", scale=2.0, n_spikes=4, spike=4.0, noise=1.0,
                                          temps="uniform:0.0:1.5", without_replacement=True)
        check_walks(rep, x, _run(sd, x, 4, True), 4, True)
    rep.finish(budget=False)


@pytest.mark.parametrize("V,dtype", [(64, "bf16"), (4099, "fp32")])
def test_tree_rr_duplicate_siblings_without_replacement(sd, V, dtype):
    """Siblings with one token are an input error only when the children were drawn
    without replacement (both kernels: 16-byte rows and scalar rows)."""
    parents = [-1, -1, 0, 0]
    x = workloads.make_tree_rr_inputs(4, V, parents, depth=2, seed=5, device=DEV, dtype=dtype,
                                      temps="const:1.0", without_replacement=True)
    x = {k: v.clone() for k, v in x.items()}
    x["node_tokens"][1, 1] = x["node_tokens"][1, 0]   # root's children
    x["node_tokens"][2, 3] = x["node_tokens"][2, 2]   # node 0's children
    x["node_tokens"][3, 2] = x["node_tokens"][3, 0]   # same token, different parents: fine
    out = _run(sd, x, 2, True)
    st = out["status"].cpu()
    assert st[1] == 32 and st[2] == 32 and (st[[0, 3]] & 0xFF == 0).all(), st
    assert (out["tokens"][1:3] == -1).all() and (out["num_accepted"][1:3] == -1).all()
    iid = _run(sd, x, 2, False)
    assert (iid["status"].cpu() & 0xFF == 0).all()


@pytest.mark.parametrize("parents,V,dtype", [
    ([], 1000, "bf16"),                                  # root only: a draw from p
    ([-1], 8, "fp32"),
    ([-1, -1, -1, -1], 64, "bf16"),                      # one node, four children
    ([-1, 0, 1, 2, 3], 4099, "fp32"),                    # a chain (odd V: scalar loads)
    ([-1, -1, 0, 0, 1, 2, 2, 5], 50000, "bf16"),
    ([-1, -1, -1, 0, 0, 0, 1, 1, 2, 3, 3, 6], 7, "fp32"),
])
def test_tree_rr_shapes(sd, parents, V, dtype):
    from oracle import specdec_oracle as so
    D = max(1, int(so.tree_depths(parents).max()) + 1) if parents else 1
    rep = Report(f"tree_rr N={len(parents)} V={V} {dtype}")
    for seed in range(4):
        x = workloads.make_tree_rr_inputs(6, V, parents, depth=D, seed=seed, device=DEV, dtype=dtype,
                                          scale=2.0, n_spikes=3, spike=3.0, noise=0.6, temps="uniform:0.0:1.5")
        check_walks(rep, x, _run(sd, x, D), D)
    rep.finish(budget=False)


@pytest.mark.parametrize("C", ["1", "2", "4", "8"])
@pytest.mark.parametrize("V,dtype", [(32008, "bf16"), (4096, "fp32"), (20004, "fp32"), (64, "bf16")])
def test_tree_rr_cluster_sizes(sd, medusa_parents, hooks, C, V, dtype):
    """Rows split across clusters of 1, 2, 4 and 8 CTAs (sizes whose slices would not fit
    or would be empty fall back to the default); short last slices at 32008 and 20004."""
    hooks(tree_cluster=int(C))
    rep = Report(f"tree_rr cluster {C} V={V} {dtype}")
    for seed in range(3):
        x = workloads.make_tree_rr_inputs(8, V, medusa_parents, depth=4, seed=40 + seed, device=DEV, dtype=dtype,
                                          scale=2.0, n_spikes=4, spike=4.0, noise=1.0, temps="uniform:0.0:1.5")
        check_walks(rep, x, _run(sd, x, 4), 4)
    rep.finish(budget=False)


def test_tree_rr_star_tree_more_children_than_the_list(sd):
    """600 children at the root (the kernel lists 256 at a time) and a few grandchildren:
    walks that reject many children refill the list; the drafter is far from the target so
    rejections are common."""
    from oracle import specdec_oracle as so
    parents = [-1] * 600 + [0, 0, 5, 599]
    rep = Report("tree_rr star, 600 children")
    for seed, dtype in ((1, "fp32"), (2, "bf16")):
        x = workloads.make_tree_rr_inputs(4, 512, parents, depth=2, seed=seed, device=DEV, dtype=dtype,
                                          scale=2.0, n_spikes=3, spike=3.0, noise=3.0, temps="const:1.0")
        check_walks(rep, x, _run(sd, x, 2), 2)
    rep.finish(budget=False)


def test_tree_rr_errors_follow_the_walk(sd):
    from oracle import specdec_oracle as so
    parents = [-1, -1, 0, 0]
    B, V, D = 10, 256, 2
    x = workloads.make_tree_rr_inputs(B, V, parents, depth=D, seed=3, device=DEV, dtype="fp32", temps="const:1.0")
    x = {k: v.clone() for k, v in x.items()}
    x["logits"][0, 0, 5] = float("nan")               # the root row
    x["logits"][1, 3, :] = float("-inf")              # node 2's row (visited only via node 0)
    x["node_tokens"][2, 1] = V                        # bad token anywhere
    x["uniforms"][3, 4] = 1.0                         # bad uniform anywhere
    x["temperatures"][4] = float("inf")
    x["draft_probs"][5, 0, 17] = -1.0                 # read only after a rejection at the root
    x["draft_probs"][6, 0, int(x["node_tokens"][6, 0])] = 0.0   # q(s) = 0 for the first child
    x["temperatures"][7] = 0.0                        # greedy
    x["draft_probs"][8, 0, int(x["node_tokens"][8, 0])] = float("nan")
    out = _run(sd, x, D)
    L, q, toks, par, T, u = (_np(x[k]) for k in KEYS)
    for b in range(B):
        o = so.verify_tree_rr_sequence(L[b], q[b], toks[b], par, float(T[b]), u[b], D)
        assert int(out["status"][b]) & 0xFF == o["status"] & 0xFF, (b, int(out["status"][b]), o["status"])
        if o["status"] & 0xFF:
            assert int(out["num_accepted"][b]) == -1 and (out["tokens"][b] == -1).all(), b
    bad_tree = torch.tensor([-1, 2, 0, 0], dtype=torch.int32, device=DEV)
    o2 = sd.verify_tree_recursive(x["logits"], x["draft_probs"], x["node_tokens"], bad_tree, x["temperatures"],
                                  x["uniforms"], D)
    assert (o2["status"] & 32).all()


def test_tree_rr_deterministic_and_fully_written(sd, medusa_parents):
    x = workloads.tree_rr_workload("tree_rr_b32_n64_v32000", medusa_parents, 3, DEV)
    B = x["logits"].shape[0]
    res = []
    for _ in range(3):
        out = {"tokens": torch.full((B, 5), 0x7F7F7F7F, dtype=torch.int32, device=DEV),
               "path": torch.full((B, 4), 0x7F7F7F7F, dtype=torch.int32, device=DEV),
               "num_accepted": torch.full((B,), 0x7F7F7F7F, dtype=torch.int32, device=DEV),
               "status": torch.full((B,), 0x7F7F7F7F, dtype=torch.int32, device=DEV)}
        sd.verify_tree_recursive(*(x[k] for k in KEYS), 4, out=out)
        torch.cuda.synchronize()
        for k, v in out.items():
            assert not (v == 0x7F7F7F7F).any(), k
        res.append({k: v.clone() for k, v in out.items()})
    for r in res[1:]:
        for k in r:
            assert torch.equal(r[k], res[0][k]), k
