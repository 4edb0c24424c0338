"""specdec_verify_chain_noalloc: chain verification that allocates nothing.

Callers under a fixed device-memory plan, plain C hosts without an allocator, and
latency-critical paths that must not let cudaMalloc synchronise the device use this entry
point; it runs on scratch memory built into the library.  This test calls it through the
C ABI twice in a row on different batches and checks every output against the workspace
entry point, specdec_verify_chain, on the same inputs.  The file is named so that pytest
collects it last; it passes alone in a fresh process as well as after the other tests.
"""
import ctypes

import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
P_TOL = 1e-6  # the tolerance the parity tests use for probabilities


def _lib(path):
    lib = ctypes.CDLL(str(path))
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    lib.specdec_verify_chain_noalloc.argtypes = [vp, i32, vp, vp, vp, vp, i32, i32, i32, vp, vp, vp, vp, vp]
    lib.specdec_verify_chain_noalloc.restype = i32
    lib.specdec_last_error.argtypes = []
    lib.specdec_last_error.restype = ctypes.c_char_p
    return lib


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, x):
    B, g1, V = x["logits"].shape
    out = {
        "tokens": torch.full((B, g1), -7, dtype=torch.int32, device=DEV),
        "num_accepted": torch.full((B,), -7, dtype=torch.int32, device=DEV),
        "p_draft": torch.full((B, g1 - 1), -7.0, device=DEV),
        "status": torch.full((B,), -7, dtype=torch.int32, device=DEV),
    }
    code = 1 if x["logits"].dtype == torch.bfloat16 else 0
    rc = lib.specdec_verify_chain_noalloc(
        _p(x["logits"]), code, _p(x["draft_probs"]), _p(x["draft_tokens"]), _p(x["temperatures"]),
        _p(x["uniforms"]), B, g1 - 1, V, _p(out["tokens"]), _p(out["num_accepted"]), _p(out["p_draft"]),
        _p(out["status"]), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, lib.specdec_last_error()
    return out


def _same(a, b):
    for k in ("tokens", "num_accepted", "status"):
        assert torch.equal(a[k], b[k]), k
    pa, pb = a["p_draft"], b["p_draft"]
    both_nan = torch.isnan(pa) & torch.isnan(pb)
    assert (both_nan | ((pa - pb).abs() <= P_TOL)).all()


@pytest.mark.parametrize("name,B", [("chain_b64_v32000", None), ("chain_b256_v128256", 32)])
def test_noalloc_matches_workspace_entry_point_twice(built_library, name, B):
    import speculative_decoding_token_temperature_gb300 as sd
    lib = _lib(built_library)
    keys = ("logits", "draft_probs", "draft_tokens", "temperatures", "uniforms")
    for r in (0, 1):  # two calls in a row on the shared scratch
        x = workloads.chain_workload(name, r, DEV, B=B)
        got = _noalloc(lib, x)
        ref = sd.verify_chain(*(x[k] for k in keys))
        torch.cuda.synchronize()
        _same(got, ref)


def test_noalloc_unaligned_rows_and_size_limit(built_library):
    import speculative_decoding_token_temperature_gb300 as sd
    lib = _lib(built_library)
    keys = ("logits", "draft_probs", "draft_tokens", "temperatures", "uniforms")
    for seed in (0, 1):
        x = workloads.make_chain_inputs(5, 3, 1001, "bf16", seed=seed, device=DEV, temps="uniform:0.0:1.2")
        got = _noalloc(lib, x)
        ref = sd.verify_chain(*(x[k] for k in keys))
        torch.cuda.synchronize()
        _same(got, ref)
    # a shape beyond the built-in scratch is refused on the host, before any launch
    big = 4096
    dummy = torch.zeros(16, device=DEV)
    rc = lib.specdec_verify_chain_noalloc(_p(dummy), 0, _p(dummy), _p(dummy), _p(dummy), _p(dummy),
                                          big, 8, 152064, _p(dummy), _p(dummy), None, None, None)
    assert rc == 5  # SPECDEC_ERR_TOO_LARGE
    assert b"built-in" in lib.specdec_last_error()
