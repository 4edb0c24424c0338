"""GPU parity of accepted-branch KV compaction (SD 20.5, "Keeping the caches consistent
after a rejection") against the oracle's gather, bit for bit, through the C ABI."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def sd(built_library):
    import speculative_decoding_token_temperature_gb300 as m
    m.load_library()
    return m


def _climbing_paths(rng, B, D, N):
    paths = np.full((B, D), -1, dtype=np.int32)
    J = np.zeros(B, dtype=np.int32)
    for b in range(B):
        j = int(rng.integers(0, D + 1))
        p = np.sort(rng.choice(N, j, replace=False)) if j else np.zeros(0, int)
        p = np.maximum(p, np.arange(j))
        while j and (np.diff(p) <= 0).any():
            p = np.sort(rng.choice(N, j, replace=False))
            p = np.maximum(p, np.arange(j))
        paths[b, :j] = p
        J[b] = j
    return paths, J


@pytest.mark.parametrize("W,dtype", [(256, torch.float32), (3, torch.bfloat16), (4096, torch.bfloat16), (1, torch.int8)])
def test_contiguous_compaction_matches_the_gather(sd, W, dtype):
    from oracle import specdec_oracle as so
    rng = np.random.default_rng(W)
    B, N, D = 8, 20, 5
    prefix = rng.integers(0, 30, B).astype(np.int32)
    S = int(prefix.max()) + N + 2
    paths, J = _climbing_paths(rng, B, D, N)
    J[3] = -1  # a failed round
    host = rng.integers(-100, 100, size=(B, S, W)).astype(np.int64)
    cache = torch.tensor(host).to(dtype).to(DEV)
    before = cache.cpu()
    res = sd.compact_kv(cache, torch.tensor(prefix, device=DEV), torch.tensor(paths, device=DEV),
                        torch.tensor(J, device=DEV))
    torch.cuda.synchronize()
    want, new_len, st = so.compact_kv(before.numpy() if dtype != torch.bfloat16 else before.view(torch.int16).numpy(),
                                      prefix, paths, J)
    got = cache.cpu()
    got = got.view(torch.int16).numpy() if dtype == torch.bfloat16 else got.numpy()
    np.testing.assert_array_equal(got, want)
    np.testing.assert_array_equal(res["new_len"].cpu().numpy(), new_len)
    np.testing.assert_array_equal(res["status"].cpu().numpy(), st)


def test_paged_compaction_matches_the_gather(sd):
    from oracle import specdec_oracle as so
    rng = np.random.default_rng(7)
    B, bs, nblk, W = 6, 8, 6, 64
    N, D = 20, 4
    table = rng.permutation(B * nblk).reshape(B, nblk).astype(np.int32)
    pool = rng.standard_normal((B * nblk, bs, W)).astype(np.float32)
    prefix = rng.integers(0, 20, B).astype(np.int32)
    paths, J = _climbing_paths(rng, B, D, N)
    cache = torch.tensor(pool, device=DEV)
    res = sd.compact_kv(cache, torch.tensor(prefix, device=DEV), torch.tensor(paths, device=DEV),
                        torch.tensor(J, device=DEV), block_table=torch.tensor(table, device=DEV))
    torch.cuda.synchronize()
    want, new_len, st = so.compact_kv(pool, prefix, paths, J, block_table=table, block_size=bs)
    np.testing.assert_array_equal(cache.cpu().numpy(), want)
    np.testing.assert_array_equal(res["new_len"].cpu().numpy(), new_len)


def test_invalid_paths_are_reported_and_left_alone(sd):
    B, S, W = 3, 16, 8
    cache = torch.arange(B * S * W, dtype=torch.float32, device=DEV).view(B, S, W)
    before = cache.clone()
    prefix = torch.tensor([0, 2, 4], dtype=torch.int32, device=DEV)
    paths = torch.tensor([[2, 1, -1], [0, 0, -1], [3, 40, -1]], dtype=torch.int32, device=DEV)  # 40 leaves the cache
    J = torch.tensor([2, 2, 2], dtype=torch.int32, device=DEV)
    res = sd.compact_kv(cache, prefix, paths, J)
    torch.cuda.synchronize()
    assert torch.equal(cache, before)
    assert (res["status"] == 32).all() and torch.equal(res["new_len"], prefix)


def test_tree_walk_then_compaction(sd):
    """The recursive-rejection walk's accepted path (from the oracle, on the same inputs)
    drives the compaction of a cache whose candidate slots hold each node's id."""
    import workloads
    from oracle import specdec_oracle as so
    parents, _, _ = so.medusa_sparse_tree(workloads.medusa_workload_accuracies(), 64)
    x = workloads.tree_rr_workload("tree_rr_b32_n64_v32000", parents, 0, "cpu")
    B, N, D, P0 = 32, 64, 4, 10
    L = x["logits"].float().numpy()
    orc = [so.verify_tree_rr_sequence(L[b], x["draft_probs"][b].numpy(), x["node_tokens"][b].numpy(), parents,
                                      float(x["temperatures"][b]), x["uniforms"][b].numpy(), D) for b in range(B)]
    paths = np.stack([o["path"] for o in orc]).astype(np.int32)
    J = np.array([o["n_accepted"] for o in orc], dtype=np.int32)
    cache = torch.zeros(B, P0 + N, 16, dtype=torch.int32)
    cache[:, P0:, 0] = torch.arange(N, dtype=torch.int32)  # slot P0 + i holds node i
    cache = cache.to(DEV)
    sd.compact_kv(cache, torch.full((B,), P0, dtype=torch.int32, device=DEV), torch.tensor(paths, device=DEV),
                  torch.tensor(J, device=DEV))
    torch.cuda.synchronize()
    c = cache.cpu().numpy()
    for b in range(B):
        assert list(c[b, P0:P0 + J[b], 0]) == list(paths[b, :J[b]])
