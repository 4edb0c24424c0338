"""Seeded synthetic inputs for speculative-decoding verification.

This module only draws random inputs; it holds none of the verification arithmetic and
imports neither the oracle nor the product library, so both sides of every parity test
see identical inputs from it.  Draft distributions q are synthesised here as
softmax(draft_logits / T), the distribution a drafter would have sampled its tokens
from; drafts are then sampled from q.

Recipes (shapes, value distributions) follow the workloads the library is measured on:

  chain_b1_v1000      B=1,   gamma=4, V=1000,   fp32 logits.  t ~ 2 N(0,1), +6 on 5 distinct ids
                      per row; d = t + 0.5 N(0,1); T = 1.
  chain_b64_v32000    B=64,  gamma=4, V=32000,  bf16.  t ~ 4 N(0,1), +10 on 8 distinct ids per
                      row; d = t + N(0,1); sequences b < 32 greedy (T = 0, q one-hot at
                      argmax d, draft = argmax d), b >= 32 at T = 0.8.
  chain_b256_v128256  B=256, gamma=7, V=128256, bf16 logits, fp32 q.  t ~ 3 N(0,1) - 1.1 ln(rank),
                      rank a random permutation of 1..V per sequence shared by its rows
                      (a Zipf(1.1) bias); d = t + 1.5 N(0,1); T = 1.
  chain_b256_v128256_s075  the same with d = t + 0.75 N(0,1).
  tree_b32_n64_v32000 B=32, 64-node Medusa tree (+ root row), V=32000, bf16, depth 4.  Per
                      sequence and head k, 10 distinct candidate ids; the node with rank path
                      (i_1..i_m) carries candidate i_m of head m.  Logits 4 N(0,1), +8 on each
                      child's token of a row independently with probability 0.5.  b < 16
                      greedy (T = 0), b >= 16 at T = 0.7.
  chain_b512_v152064  B=512, gamma=8, V=152064, fp32.  t ~ 3 N(0,1) - ln(rank); sigma_b ~ U(0.5,
                      2.5); d = t + sigma_b N(0,1); T_b ~ U(0, 1.2), T_b < 1e-3 greedy.

Uniforms are U[0,1) of shape [B, gamma+1] (chain) or [B, depth+1] (tree).  The seed of
round r of a workload is 1000 * (workload number) + r.
"""
from __future__ import annotations

import torch

GREEDY_BELOW = 1e-3

CHAIN_WORKLOADS = {
    "chain_b1_v1000": dict(number=1, B=1, gamma=4, V=1000, dtype="fp32", recipe="spikes",
                           scale=2.0, n_spikes=5, spike=6.0, noise=0.5, temps="const:1.0"),
    "chain_b64_v32000": dict(number=2, B=64, gamma=4, V=32000, dtype="bf16", recipe="spikes",
                             scale=4.0, n_spikes=8, spike=10.0, noise=1.0, temps="half_greedy:0.8"),
    "chain_b256_v128256": dict(number=3, B=256, gamma=7, V=128256, dtype="bf16", recipe="zipf",
                               scale=3.0, zipf_s=1.1, noise=1.5, temps="const:1.0"),
    "chain_b256_v128256_s075": dict(number=6, B=256, gamma=7, V=128256, dtype="bf16", recipe="zipf",
                                    scale=3.0, zipf_s=1.1, noise=0.75, temps="const:1.0"),
    "chain_b512_v152064": dict(number=5, B=512, gamma=8, V=152064, dtype="fp32", recipe="zipf",
                               scale=3.0, zipf_s=1.0, noise="uniform:0.5:2.5", temps="uniform:0.0:1.2"),
}

TREE_RR_WORKLOADS = {
    # the Medusa sparse tree's topology (64 nodes, depth 4), tokens drafted i.i.d. per node
    "tree_rr_b32_n64_v32000": dict(number=7, B=32, V=32000, dtype="bf16", depth=4, recipe="spikes",
                                   scale=4.0, n_spikes=8, spike=8.0, noise=1.0, temps="uniform:0.0:1.2"),
}

TREE_WORKLOADS = {
    "tree_b32_n64_v32000": dict(number=4, B=32, V=32000, dtype="bf16", depth=4, top=10,
                                scale=4.0, spike=8.0, spike_prob=0.5, temps="half_greedy:0.7"),
}

# The assumed per-head top-k accuracies of the tree workload: a_k^(i) = 0.6 * 0.75^(i-1) *
# 0.85^(k-1), head k = 1..4, rank i = 1..10, as exact fractions.
def medusa_workload_accuracies(heads: int = 4, top: int = 10):
    from fractions import Fraction
    return [[Fraction(3, 5) * Fraction(3, 4) ** (i - 1) * Fraction(17, 20) ** (k - 1)
             for i in range(1, top + 1)] for k in range(1, heads + 1)]


def seed_for(workload_number: int, round_idx: int) -> int:
    return 1000 * workload_number + round_idx


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _temperatures(spec: str, B: int, g, device):
    kind, _, rest = spec.partition(":")
    if kind == "const":
        return torch.full((B,), float(rest), dtype=torch.float32, device=device)
    if kind == "half_greedy":
        T = torch.full((B,), float(rest), dtype=torch.float32, device=device)
        T[: B // 2] = 0.0
        return T
    if kind == "uniform":
        lo, hi = (float(x) for x in rest.split(":"))
        return lo + (hi - lo) * torch.rand(B, generator=g, device=device)
    raise ValueError(spec)


def _noise_scale(spec, B, g, device):
    if isinstance(spec, (int, float)):
        return torch.full((B, 1, 1), float(spec), device=device)
    kind, lo, hi = spec.split(":")
    assert kind == "uniform"
    return (float(lo) + (float(hi) - float(lo)) * torch.rand(B, generator=g, device=device)).view(B, 1, 1)


def _spike_ids(rows: int, V: int, k: int, g, device):
    """k distinct random ids in [0, V) per row (top-k of i.i.d. random keys)."""
    keys = torch.rand(rows, V, generator=g, device=device)
    return torch.topk(keys, k, dim=1).indices


def make_chain_inputs(B: int, gamma: int, V: int, dtype: str = "bf16", *, seed: int = 0,
                      device="cpu", recipe: str = "spikes", scale: float = 2.0,
                      n_spikes: int = 5, spike: float = 6.0, zipf_s: float = 1.0,
                      noise=0.5, temps: str = "const:1.0", q_dtype=torch.float32) -> dict:
    """Seeded chain-verification inputs.

    Returns logits [B, gamma+1, V] (bf16 or fp32), draft_probs [B, gamma, V] (fp32),
    draft_tokens [B, gamma] (int32), temperatures [B] (fp32), uniforms [B, gamma+1] (fp32).
    """
    g = _gen(device, seed)
    rows = B * (gamma + 1)
    t = scale * torch.randn(B, gamma + 1, V, generator=g, device=device)
    if recipe == "spikes":
        ids = _spike_ids(rows, V, n_spikes, g, device)
        t.view(rows, V).scatter_add_(1, ids, torch.full(ids.shape, spike, device=device))
    elif recipe == "zipf":
        perm = torch.argsort(torch.rand(B, V, generator=g, device=device), dim=1)
        bias = -zipf_s * torch.log((perm + 1).to(torch.float32))
        t += bias.view(B, 1, V)
        del perm, bias
    else:
        raise ValueError(recipe)
    sigma = _noise_scale(noise, B, g, device)
    d = t[:, :gamma, :] + sigma * torch.randn(B, gamma, V, generator=g, device=device)
    T = _temperatures(temps, B, g, device)
    greedy = T < GREEDY_BELOW
    Tq = torch.where(greedy, torch.ones_like(T), T).view(B, 1, 1)
    q = torch.softmax(d / Tq, dim=-1)
    if greedy.any():
        hot = torch.zeros_like(q[greedy])
        hot.scatter_(2, d[greedy].argmax(dim=-1, keepdim=True), 1.0)
        q[greedy] = hot
    del d
    drafts = torch.multinomial(q.view(B * gamma, V), 1, generator=g).view(B, gamma)
    u = torch.rand(B, gamma + 1, generator=g, device=device)
    logits = t.to(torch.bfloat16) if dtype == "bf16" else t
    return {
        "logits": logits.contiguous(),
        "draft_probs": q.to(q_dtype).contiguous(),
        "draft_tokens": drafts.to(torch.int32).contiguous(),
        "temperatures": T.contiguous(),
        "uniforms": u.contiguous(),
    }


def chain_workload(name: str, round_idx: int = 0, device="cpu", B: int | None = None) -> dict:
    """Inputs of a named chain workload (optionally only its first B sequences' shape)."""
    w = dict(CHAIN_WORKLOADS[name])
    number = w.pop("number")
    Bw = w.pop("B")
    return make_chain_inputs(B or Bw, w.pop("gamma"), w.pop("V"), w.pop("dtype"),
                             seed=seed_for(number, round_idx), device=device, **w)


def make_tree_inputs(B: int, V: int, parents, paths, *, depth: int, seed: int = 0, device="cpu",
                     dtype: str = "bf16", top: int = 10, scale: float = 4.0, spike: float = 8.0,
                     spike_prob: float = 0.5, temps: str = "half_greedy:0.7") -> dict:
    """Seeded tree-verification inputs for a given topology.

    parents [N] and paths (rank tuples, 0-based, one per node) describe the tree.
    Returns logits [B, N+1, V], node_tokens [B, N] int32, parents [N] int32,
    temperatures [B], uniforms [B, depth+1].
    """
    g = _gen(device, seed)
    N = len(parents)
    heads = max(len(p) for p in paths)
    cand = _spike_ids(B * heads, V, top, g, device).view(B, heads, top)
    last_rank = torch.tensor([p[-1] for p in paths], device=device)
    head_of = torch.tensor([len(p) - 1 for p in paths], device=device)
    node_tokens = cand[:, head_of, last_rank]                       # [B, N]
    t = scale * torch.randn(B, N + 1, V, generator=g, device=device)
    parent_row = torch.tensor([0 if a < 0 else 1 + a for a in parents], device=device)
    coin = torch.rand(B, N, generator=g, device=device) < spike_prob
    bump = torch.where(coin, torch.full((B, N), spike, device=device), torch.zeros(B, N, device=device))
    flat = t.view(B * (N + 1), V)
    row_idx = (torch.arange(B, device=device).view(B, 1) * (N + 1) + parent_row.view(1, N)).reshape(-1)
    flat.index_put_((row_idx, node_tokens.reshape(-1)), bump.reshape(-1), accumulate=True)
    T = _temperatures(temps, B, g, device)
    u = torch.rand(B, depth + 1, generator=g, device=device)
    logits = t.to(torch.bfloat16) if dtype == "bf16" else t
    return {
        "logits": logits.contiguous(),
        "node_tokens": node_tokens.to(torch.int32).contiguous(),
        "parents": torch.tensor(list(parents), dtype=torch.int32, device=device),
        "temperatures": T.contiguous(),
        "uniforms": u.contiguous(),
    }


def make_tree_rr_inputs(B: int, V: int, parents, *, depth: int, seed: int = 0, device="cpu",
                        dtype: str = "bf16", recipe: str = "spikes", scale: float = 4.0, n_spikes: int = 8,
                        spike: float = 8.0, noise=1.0, temps: str = "const:1.0",
                        without_replacement: bool = False) -> dict:
    """Seeded inputs for sampled tree verification with per-node drafting distributions.

    Target logits per node (row 0: the root), a drafter that sees the target logits plus
    Gaussian noise (q = softmax((l + noise) / T), one-hot at its argmax for a greedy
    sequence), and every node's token drawn from its parent's q row, independently for
    siblings -- or, with without_replacement, a node's children drawn in index order
    without replacement from its q row (distinct tokens; a greedy sequence's one-hot row
    gets a small floor first, since its walk does not use q).  Returns logits [B, N+1, V],
    draft_probs [B, N+1, V] fp32, node_tokens [B, N] int32, parents [N] int32,
    temperatures [B], uniforms [B, N+1].
    """
    g = _gen(device, seed)
    N = len(parents)
    rows = B * (N + 1)
    t = scale * torch.randn(B, N + 1, V, generator=g, device=device)
    if recipe == "spikes":
        ids = _spike_ids(rows, V, min(n_spikes, V), g, device)
        t.view(rows, V).scatter_add_(1, ids, torch.full(ids.shape, spike, device=device))
    else:
        raise ValueError(recipe)
    sigma = _noise_scale(noise, B, g, device)
    d = t + sigma * torch.randn(B, N + 1, V, generator=g, device=device)
    T = _temperatures(temps, B, g, device)
    greedy = T < GREEDY_BELOW
    Tq = torch.where(greedy, torch.ones_like(T), T).view(B, 1, 1)
    q = torch.softmax(d / Tq, dim=-1)
    if greedy.any():
        hot = torch.zeros_like(q[greedy])
        hot.scatter_(2, d[greedy].argmax(dim=-1, keepdim=True), 1.0)
        q[greedy] = hot
    del d
    parent_row = torch.tensor([0 if a < 0 else 1 + a for a in parents], dtype=torch.long, device=device)
    if N and without_replacement:
        node_tokens = torch.zeros(B, N, dtype=torch.long, device=device)
        for a in sorted(set(parents)):
            kids = [j for j in range(N) if parents[j] == a]
            qa = q[:, 0 if a < 0 else 1 + a, :]
            qa = torch.where(greedy.view(B, 1), qa + 1e-6, qa)
            node_tokens[:, kids] = torch.multinomial(qa, len(kids), replacement=False, generator=g)
    elif N:
        qp = q[:, parent_row, :].reshape(B * N, V)
        node_tokens = torch.multinomial(qp, 1, generator=g).view(B, N)
    else:
        node_tokens = torch.zeros(B, 0, dtype=torch.long, device=device)
    u = torch.rand(B, N + 1, generator=g, device=device)
    logits = t.to(torch.bfloat16) if dtype == "bf16" else t
    return {
        "logits": logits.contiguous(),
        "draft_probs": q.contiguous(),
        "node_tokens": node_tokens.to(torch.int32).contiguous(),
        "parents": torch.tensor(list(parents), dtype=torch.int32, device=device),
        "temperatures": T.contiguous(),
        "uniforms": u.contiguous(),
    }


def tree_rr_workload(name: str, parents, round_idx: int = 0, device="cpu",
                     without_replacement: bool = False) -> dict:
    w = dict(TREE_RR_WORKLOADS[name])
    number = w.pop("number")
    return make_tree_rr_inputs(w.pop("B"), w.pop("V"), parents, depth=w.pop("depth"),
                               seed=seed_for(number, round_idx), device=device,
                               without_replacement=without_replacement, **w)


def tree_workload(name: str, parents, paths, round_idx: int = 0, device="cpu") -> dict:
    w = dict(TREE_WORKLOADS[name])
    number = w.pop("number")
    return make_tree_inputs(w.pop("B"), w.pop("V"), parents, paths, depth=w.pop("depth"),
                            seed=seed_for(number, round_idx), device=device, **w)
