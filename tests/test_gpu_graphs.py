"""The library's calls inside CUDA graphs: a serving loop captures a verification step once
and replays it, so every entry point must issue only stream-ordered work (no synchronising
call, no host read of device data) and give the same outputs when replayed as when called
directly.  Each case captures the call on a side stream, replays it, and compares every
output with a direct call on the same inputs, bit for bit."""
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module")
def sd(built_library):
    import speculative_decoding_token_temperature_gb300 as m
    m.load_library()
    return m


def _captured(fn, out_like):
    """fn(out, stream) issued inside a CUDA graph; returns the outputs of one replay."""
    out = {k: torch.full_like(v, 0x55) for k, v in out_like.items()}
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn(out, side)  # warm-up outside the capture (one-time function attributes)
        torch.cuda.synchronize()
        for v in out.values():
            v.fill_(0x55)
        with torch.cuda.graph(g, stream=side):
            fn(out, side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for v in out.values():
        v.fill_(0x55)
    g.replay()
    torch.cuda.synchronize()
    return out


def _same(a, b):
    """Bit-for-bit, NaN fills included."""
    for k in a:
        x, y = a[k], b[k]
        if x.dtype == torch.float32:
            x, y = x.view(torch.int32), y.view(torch.int32)
        assert torch.equal(x, y), k


@pytest.mark.parametrize("name", ["chain_b64_v32000", "chain_b256_v128256"])
def test_chain_in_graph(sd, name):
    x = workloads.chain_workload(name, 1, DEV)
    keys = ("logits", "draft_probs", "draft_tokens", "temperatures", "uniforms")
    ref = sd.verify_chain(*(x[k] for k in keys))
    torch.cuda.synchronize()
    got = _captured(lambda out, s: sd.verify_chain(*(x[k] for k in keys), out=out, stream=s), ref)
    _same(ref, got)


def test_block_in_graph(sd):
    x = workloads.chain_workload("chain_b64_v32000", 2, DEV)
    keys = ("logits", "draft_probs", "draft_tokens", "temperatures", "uniforms")
    ref = sd.verify_block(*(x[k] for k in keys))
    torch.cuda.synchronize()
    got = _captured(lambda out, s: sd.verify_block(*(x[k] for k in keys), out=out, stream=s), ref)
    _same(ref, got)


def test_tree_walks_and_compaction_in_graph(sd):
    from oracle import specdec_oracle as so  # the tree topology only
    parents, paths, _ = so.medusa_sparse_tree(workloads.medusa_workload_accuracies(), 64)
    t = workloads.tree_workload("tree_b32_n64_v32000", parents, paths, 1, DEV)
    tk = ("logits", "node_tokens", "parents", "temperatures", "uniforms")
    ref = sd.verify_tree(*(t[k] for k in tk), 4)
    torch.cuda.synchronize()
    _same(ref, _captured(lambda out, s: sd.verify_tree(*(t[k] for k in tk), 4, out=out, stream=s), ref))

    r = workloads.tree_rr_workload("tree_rr_b32_n64_v32000", parents, 1, DEV)
    rk = ("logits", "draft_probs", "node_tokens", "parents", "temperatures", "uniforms")
    ref = sd.verify_tree_recursive(*(r[k] for k in rk), 4)
    torch.cuda.synchronize()
    _same(ref, _captured(lambda out, s: sd.verify_tree_recursive(*(r[k] for k in rk), 4, out=out, stream=s), ref))

    # compaction along the walks: replaying the captured call moves the same slots
    B, N = 32, len(parents)
    gen = torch.Generator(device=DEV).manual_seed(3)
    base = torch.randn(B, 8 + N, 256, generator=gen, device=DEV).to(torch.bfloat16)
    prefix = torch.full((B,), 8, dtype=torch.int32, device=DEV)
    want = base.clone()
    sd.compact_kv(want, prefix, ref["path"], ref["num_accepted"])
    got = base.clone()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            sd.compact_kv(got, prefix, ref["path"], ref["num_accepted"], stream=side)
    torch.cuda.current_stream().wait_stream(side)
    got.copy_(base)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(got, want)
