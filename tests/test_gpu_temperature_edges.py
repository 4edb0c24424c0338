"""Temperatures at the edges, through the C ABI, against the fp64 oracle: exactly at the
greedy threshold (1e-3 in float32: sampled), one float32 step below it (greedy), zero,
tiny but sampled (a nearly one-hot target), and very large (a nearly uniform target).
The oracle and every kernel must take the same greedy-or-sampled decision for each
sequence (the threshold test is `T < 1e-3`, in the precision of the input), and sampled
sequences follow the parity rules of tests/parity.py."""
import numpy as np
import pytest
import torch

import workloads
from parity import ParityReport, check_chain, run_oracle_chain

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
KEYS = ("logits", "draft_probs", "draft_tokens", "temperatures", "uniforms")

T_EDGES = np.array([1e-3, np.nextafter(np.float32(1e-3), np.float32(0)), 0.0, 2e-3, 1e4, 1.0], dtype=np.float32)


@pytest.fixture(scope="module")
def sd(built_library):
    import speculative_decoding_token_temperature_gb300 as m
    m.load_library()
    return m


def _np(t):
    return (t.float() if t.dtype == torch.bfloat16 else t).detach().cpu().numpy()


def _inputs(V, dtype, seed):
    B = len(T_EDGES)
    x = workloads.make_chain_inputs(B, 4, V, dtype, seed=seed, device=DEV, recipe="spikes", scale=2.0,
                                    n_spikes=3, spike=4.0, noise=0.5, temps="const:1.0")
    x = dict(x)
    x["temperatures"] = torch.tensor(T_EDGES, device=DEV)
    return x


def test_threshold_reading_in_float32():
    # the float32 value of 1e-3 lies above the float64 threshold, one step below it under
    from oracle import specdec_oracle as so
    assert not (float(T_EDGES[0]) < so.GREEDY_T) and float(T_EDGES[1]) < so.GREEDY_T


@pytest.mark.parametrize("V,dtype", [(4096, "fp32"), (32000, "bf16")])
@pytest.mark.parametrize("rule", ["chain", "block"])
def test_chain_and_block_at_temperature_edges(sd, V, dtype, rule):
    rep = ParityReport(f"{rule} temperature edges V={V} {dtype}")
    for seed in range(4):
        x = _inputs(V, dtype, seed)
        call = sd.verify_chain if rule == "chain" else sd.verify_block
        out = call(*(x[k] for k in KEYS))
        torch.cuda.synchronize()
        gpu = {k: _np(v) for k, v in out.items()}
        orc = run_oracle_chain(*(_np(x[k]) for k in KEYS), gpu["tokens"], gpu["num_accepted"], workers=1,
                               mode=rule)
        for b, o in enumerate(orc):
            assert o["greedy"] == bool(T_EDGES[b] < np.float32(1e-3)), (b, T_EDGES[b])
        check_chain(rep, gpu, orc, _np(x["uniforms"]), rule=rule)
    assert not rep.failures, rep.failures[:5]
    assert rep.flagged == 0, rep.summary()


def test_tree_walks_at_temperature_edges(sd):
    from oracle import specdec_oracle as so
    parents = [-1, -1, 0, 0, 1, 2]
    B, V, D = len(T_EDGES), 4096, 3
    for seed in range(4):
        x = workloads.make_tree_rr_inputs(B, V, parents, depth=D, seed=seed, device=DEV, dtype="bf16", scale=2.0,
                                          n_spikes=3, spike=4.0, noise=0.5, temps="const:1.0")
        x = dict(x)
        x["temperatures"] = torch.tensor(T_EDGES, device=DEV)
        keys = ("logits", "draft_probs", "node_tokens", "parents", "temperatures", "uniforms")
        out = sd.verify_tree_recursive(*(x[k] for k in keys), D)
        med = sd.verify_tree(x["logits"], x["node_tokens"], x["parents"], x["temperatures"],
                             x["uniforms"][:, :D + 1].contiguous(), D)
        torch.cuda.synchronize()
        L, q, toks, T, u = (_np(x[k]) for k in ("logits", "draft_probs", "node_tokens", "temperatures", "uniforms"))
        for b in range(B):
            o = so.verify_tree_rr_sequence(L[b], q[b], toks[b], parents, float(T[b]), u[b], D)
            assert o["greedy"] == bool(T_EDGES[b] < np.float32(1e-3))
            if o["greedy"]:  # greedy walks are exact
                assert _np(out["tokens"])[b].tolist() == o["tokens"].tolist(), (b, T_EDGES[b])
                assert int(out["num_accepted"][b]) == o["n_accepted"]
            if o["greedy"]:  # the Medusa walk: greedy walks exact as well
                m = so.verify_tree_sequence(L[b], toks[b], parents, float(T[b]), u[b][:D + 1], D)
                assert _np(med["tokens"])[b].tolist() == m["tokens"].tolist(), (b, T_EDGES[b])
