"""Chain verification reading logits and draft probabilities in place from pinned host
memory (specdec.h, "Host-resident rows"): the left-to-right kernel fetches only the rows
the round needs (SD 20.5, "A whole round of speculative sampling": rows after the first
rejection are never needed) over the host link.  The arithmetic is the device-memory
kernel's, so the outputs must be the same bits as with device inputs; the device path is
held to the oracle by tests/test_gpu_chain.py, and one case here is checked against the
oracle directly."""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from parity import ParityReport, check_chain, run_oracle_chain

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
KEYS = ("logits", "draft_probs", "draft_tokens", "temperatures", "uniforms")


@pytest.fixture(scope="module")
def sd(built_library):
    import speculative_decoding_token_temperature_gb300 as m
    m.load_library()
    return m


def _np(t):
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.detach().cpu().numpy()


def _pinned(x):
    return {k: v.cpu().pin_memory() for k, v in x.items()}


def _same(a, b):
    for k in a:
        av, bv = a[k].cpu().float(), b[k].cpu().float()
        assert torch.equal(torch.nan_to_num(av, nan=-7.0), torch.nan_to_num(bv, nan=-7.0)), k


def test_host_rows_match_device_rows(sd):
    for seed in range(3):
        x = workloads.chain_workload("chain_b64_v32000", seed, DEV)
        dev_out = sd.verify_chain(*(x[k] for k in KEYS))
        h = _pinned(x)
        host_out = sd.verify_chain(*(h[k] for k in KEYS))
        assert host_out["tokens"].device.type == "cpu"
        _same(dev_out, host_out)


def test_host_rows_oracle(sd):
    rep = ParityReport("chain_b64_v32000 from pinned host rows")
    x = _pinned(workloads.chain_workload("chain_b64_v32000", 11, "cpu"))
    out = sd.verify_chain(*(x[k] for k in KEYS))
    gpu = {k: _np(v) for k, v in out.items()}
    orc = run_oracle_chain(*(_np(x[k]) for k in KEYS), gpu["tokens"], gpu["num_accepted"])
    check_chain(rep, gpu, orc, _np(x["uniforms"]))
    assert not rep.failures, rep.failures[:10]


def test_host_rows_full_size(sd):
    x = workloads.chain_workload("chain_b256_v128256", 2, DEV)
    dev_out = sd.verify_chain(*(x[k] for k in KEYS))
    h = _pinned(x)
    del x
    torch.cuda.empty_cache()
    _same(dev_out, sd.verify_chain(*(h[k] for k in KEYS)))


@pytest.mark.parametrize("B,gamma,V,dtype", [
    (5, 3, 1001, "fp32"), (4, 4, 1000, "bf16"), (3, 2, 16384 + 8, "bf16"), (7, 5, 50000, "bf16"),
    (2, 16, 4099, "bf16"), (1, 1, 8, "fp32"), (2, 40, 64, "fp32"),
])
def test_host_rows_ragged(sd, B, gamma, V, dtype):
    """Aligned rows are read in place; unaligned rows (V = 4099 bf16) and g + 1 > 32 are
    refused by the library and copied by the binding instead."""
    for seed in range(2):
        x = workloads.make_chain_inputs(B, gamma, V, dtype, seed=seed, device=DEV,
                                        recipe="spikes", scale=2.0, n_spikes=min(3, V), spike=4.0,
                                        noise=0.7, temps="uniform:0.0:1.5")
        _same(sd.verify_chain(*(x[k] for k in KEYS)), sd.verify_chain(*(_pinned(x)[k] for k in KEYS)))


def test_host_rows_greedy_and_varlen(sd):
    x = workloads.chain_workload("chain_b64_v32000", 4, DEV)
    h = _pinned(x)
    _same(sd.verify_greedy(x["logits"], x["draft_tokens"]), sd.verify_greedy(h["logits"], h["draft_tokens"]))
    gm = torch.from_numpy(np.random.default_rng(4).integers(0, 8, 64).astype(np.int32))
    _same(sd.verify_chain_varlen(*(x[k] for k in KEYS), gm.to(DEV)),
          sd.verify_chain_varlen(*(h[k] for k in KEYS), gm))


def test_pageable_host_rows_are_refused(sd):
    """The C ABI refuses pageable host memory before launching anything."""
    lib = sd.load_library()
    B, g, V = 2, 2, 64
    x = workloads.make_chain_inputs(B, g, V, "fp32", seed=0, device=DEV, temps="const:1.0")
    pageable = torch.zeros(B, g + 1, V)  # not pinned
    assert not pageable.is_pinned()
    ws = torch.empty(int(lib.specdec_chain_workspace_bytes(B, g, V, sd.F32)), dtype=torch.uint8, device=DEV)
    toks = torch.empty(B, g + 1, dtype=torch.int32, device=DEV)
    J = torch.empty(B, dtype=torch.int32, device=DEV)
    p = ctypes.c_void_p
    rc = lib.specdec_verify_chain(p(pageable.data_ptr()), sd.F32, p(x["draft_probs"].data_ptr()),
                                  p(x["draft_tokens"].data_ptr()), p(x["temperatures"].data_ptr()),
                                  p(x["uniforms"].data_ptr()), B, g, V, p(toks.data_ptr()), p(J.data_ptr()),
                                  None, None, p(ws.data_ptr()), ctypes.c_size_t(ws.numel()), None)
    assert rc == 1  # SPECDEC_ERR_INVALID_ARG
    assert b"pinned" in lib.specdec_last_error()


def _abi_chain(sd, x, ws_bytes):
    """specdec_verify_chain through the C ABI with a workspace of the given size."""
    lib = sd.load_library()
    B, g1, V = x["logits"].shape
    g = g1 - 1
    code = sd.BF16 if x["logits"].dtype == torch.bfloat16 else sd.F32
    ws = torch.empty(int(ws_bytes), dtype=torch.uint8, device=DEV)
    out = {"tokens": torch.full((B, g1), -9, dtype=torch.int32, device=DEV),
           "num_accepted": torch.full((B,), -9, dtype=torch.int32, device=DEV),
           "p_draft": torch.full((B, g), -9.0, dtype=torch.float32, device=DEV),
           "status": torch.full((B,), -9, dtype=torch.int32, device=DEV)}
    p = ctypes.c_void_p
    d = {k: (v if v.device.type == "cpu" else v.to(DEV)) for k, v in x.items()}
    for k in ("draft_tokens", "temperatures", "uniforms"):
        d[k] = x[k].to(DEV)
    rc = lib.specdec_verify_chain(p(d["logits"].data_ptr()), code, p(d["draft_probs"].data_ptr()),
                                  p(d["draft_tokens"].data_ptr()), p(d["temperatures"].data_ptr()),
                                  p(d["uniforms"].data_ptr()), B, g, V, p(out["tokens"].data_ptr()),
                                  p(out["num_accepted"].data_ptr()), p(out["p_draft"].data_ptr()),
                                  p(out["status"].data_ptr()), p(ws.data_ptr()), ctypes.c_size_t(ws.numel()),
                                  p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, lib.specdec_last_error()
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("case", [
    ("chain_b256_v128256", 0), ("chain_b256_v128256", 1), ("chain_b256_v128256_s075", 0),
    ("chain_b64_v32000", 3), (300, 3, 4096, "bf16"), (9, 7, 50000, "fp32"), (4, 31, 8192, "bf16"),
])
def test_host_rows_device_copy_same_bits(sd, case):
    """With host logits and the larger workspace (specdec_chain_host_workspace_bytes) the
    kernel keeps a device copy of each sequence's latest row and draws read it; with the
    plain workspace they read the host row again.  Both give the device-input bits, for
    queued and immediate draws, rows computed ahead and mixed greedy/sampled sequences."""
    lib = sd.load_library()
    if isinstance(case[0], str):
        x = {k: v.cpu() for k, v in workloads.chain_workload(case[0], case[1], DEV).items()}
    else:
        B, g, V, dt = case
        x = workloads.make_chain_inputs(B, g, V, dt, seed=5, device=DEV, recipe="spikes", scale=2.0,
                                        n_spikes=3, spike=4.0, noise=0.6, temps="uniform:0.0:1.5")
        x = {k: v.cpu() for k, v in x.items()}
    B, g1, V = x["logits"].shape
    code = sd.BF16 if x["logits"].dtype == torch.bfloat16 else sd.F32
    small = lib.specdec_chain_workspace_bytes(B, g1 - 1, V, code)
    big = lib.specdec_chain_host_workspace_bytes(B, g1 - 1, V, code)
    assert big > small
    ref = _abi_chain(sd, {k: v.to(DEV) for k, v in x.items()}, small)
    h = _pinned(x)
    _same(ref, _abi_chain(sd, h, big))    # device copy of the drawn rows
    _same(ref, _abi_chain(sd, h, small))  # drawn rows read from the host again
    # logits on the host with q on the device (the copy is used), and q alone on the host
    # (it is not: nothing of the logits sits on the host)
    _same(ref, _abi_chain(sd, {**h, "draft_probs": x["draft_probs"].to(DEV)}, big))
    _same(ref, _abi_chain(sd, {**h, "logits": x["logits"].to(DEV)}, big))


def test_host_inputs_on_the_callers_stream(sd):
    """Host inputs with a `stream=` other than the current one: the binding's copies run on
    that stream, so a stream kept busy before the call still sees the inputs land before
    the kernel and the outputs read after it (a clock spin of a few ms holds it back)."""
    x = workloads.chain_workload("chain_b64_v32000", 5, DEV)
    ref = sd.verify_chain(*(x[k] for k in KEYS))
    ref_g = sd.verify_greedy(x["logits"], x["draft_tokens"])
    side = torch.cuda.Stream()
    for h in ({k: v.cpu() for k, v in x.items()}, _pinned(x)):  # copied rows, rows read in place
        with torch.cuda.stream(side):
            torch.cuda._sleep(20_000_000)
        _same(ref, sd.verify_chain(*(h[k] for k in KEYS), stream=side))
        with torch.cuda.stream(side):
            torch.cuda._sleep(20_000_000)
        _same(ref_g, sd.verify_greedy(h["logits"], h["draft_tokens"], stream=side))
    torch.cuda.synchronize()
