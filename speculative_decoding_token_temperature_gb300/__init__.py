"""GB300 (sm_103a) speculative-decoding verification.

A thin ctypes binding over the C ABI in ``include/specdec.h`` (``libspecdec.so``, built
in-tree by ``build.py``).  The binding only marshals arguments: it checks shapes and
dtypes, passes raw device pointers and the current CUDA stream to the library, and, for
tensors that live on the host, copies inputs to the device and results back.  Every
step of verification runs in the library's CUDA kernels; there is no CPU fallback, and
calling without the compiled library raises.
"""
from __future__ import annotations

import contextlib
import ctypes
from pathlib import Path

import torch

__all__ = [
    "SpecdecError", "verify_chain", "verify_greedy", "verify_tree", "build_tree_mask",
    "chain_workspace_bytes", "library_path", "load_library", "KernelTimer",
    "F32", "BF16", "GREEDY_TEMPERATURE",
]

F32, BF16 = 0, 1
GREEDY_TEMPERATURE = 1e-3
STATUS_TIMEOUT = 128
TREE_WITHOUT_REPLACEMENT = 1  # specdec_verify_tree_recursive: children drawn without replacement

# Test hooks of the library (specdec_set_test_hook): the library's own tests and sweeps.
HOOK_CHAIN_ALL_ROWS, HOOK_BLOCK_TWO_PASS, HOOK_TREE_CLUSTER, HOOK_CHAIN_DROP_DRAWS, HOOK_QUEUE_WAIT_US = range(5)

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_WORKSPACE = 0, 1, 2, 3, 4
_ERR_NAMES = {1: "invalid argument", 2: "unsupported size", 3: "CUDA launch error",
              4: "workspace too small"}

STATUS_BAD_LOGIT = 1
STATUS_EMPTY_ROW = 2
STATUS_BAD_TOKEN = 4
STATUS_BAD_PROB = 8
STATUS_BAD_UNIFORM = 16
STATUS_BAD_TREE = 32
STATUS_BAD_TEMPERATURE = 64
STATUS_TIMEOUT = 128
STATUS_ERROR_MASK = 0xFF
STATUS_ZERO_Q = 256
STATUS_ZERO_RESIDUAL = 512

KERNEL_NAMES = ("chain_stats", "chain_sample", "tree_walk", "tree_mask", "chain_decide", "chain_finish",
                "chain_seq", "block_decide", "block_finish", "block_fused", "tree_rr", "gumbel",
                "gumbel_draft", "kv_compact")


class SpecdecError(RuntimeError):
    pass


_LIB = None


def library_path() -> Path:
    return Path(__file__).resolve().with_name("libspecdec.so")


def load_library():
    """Load libspecdec.so (raises if it has not been built)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = library_path()
    if not path.exists():
        raise SpecdecError(f"{path.name} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(str(path))
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.specdec_chain_workspace_bytes.argtypes = [i32, i32, i32, i32]
    lib.specdec_chain_workspace_bytes.restype = sz
    lib.specdec_chain_host_workspace_bytes.argtypes = [i32, i32, i32, i32]
    lib.specdec_chain_host_workspace_bytes.restype = sz
    lib.specdec_greedy_workspace_bytes.argtypes = [i32, i32, i32, i32]
    lib.specdec_greedy_workspace_bytes.restype = sz
    lib.specdec_block_workspace_bytes.argtypes = [i32, i32, i32, i32]
    lib.specdec_block_workspace_bytes.restype = sz
    lib.specdec_tree_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
    lib.specdec_tree_workspace_bytes.restype = sz
    lib.specdec_verify_chain.argtypes = [vp, i32, vp, vp, vp, vp, i32, i32, i32, vp, vp, vp, vp, vp, sz, vp]
    lib.specdec_verify_chain.restype = i32
    lib.specdec_verify_chain_varlen.argtypes = [vp, i32, vp, vp, vp, vp, vp, i32, i32, i32, vp, vp, vp, vp, vp, sz,
                                                vp]
    lib.specdec_verify_chain_varlen.restype = i32
    lib.specdec_verify_block.argtypes = [vp, i32, vp, vp, vp, vp, i32, i32, i32, vp, vp, vp, vp, vp, sz, vp]
    lib.specdec_verify_block.restype = i32
    lib.specdec_verify_greedy.argtypes = [vp, i32, vp, i32, i32, i32, vp, vp, vp, vp, sz, vp]
    lib.specdec_verify_greedy.restype = i32
    lib.specdec_verify_tree.argtypes = [vp, i32, vp, vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, sz, vp]
    lib.specdec_verify_tree.restype = i32
    lib.specdec_verify_tree_recursive.argtypes = [vp, i32, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp]
    lib.specdec_verify_tree_recursive.restype = i32
    u64 = ctypes.c_uint64
    lib.specdec_gumbel_workspace_bytes.argtypes = [i32, i32]
    lib.specdec_gumbel_workspace_bytes.restype = sz
    lib.specdec_verify_gumbel.argtypes = [vp, i32, vp, vp, u64, i32, i32, i32, vp, vp, vp, vp, sz, vp]
    lib.specdec_verify_gumbel.restype = i32
    lib.specdec_gumbel_draft.argtypes = [vp, u64, i32, i32, i32, vp, vp]
    lib.specdec_gumbel_draft.restype = i32
    lib.specdec_gumbel_noise.argtypes = [u64, i32, i32, i32, vp, vp]
    lib.specdec_gumbel_noise.restype = i32
    i64 = ctypes.c_int64
    lib.specdec_compact_kv.argtypes = [vp, i64, i64, i64, i64, vp, i32, i32, i64, i32, vp, vp, i32, vp, vp, vp, vp]
    lib.specdec_compact_kv.restype = i32
    lib.specdec_build_tree_mask.argtypes = [vp, i32, i32, vp, vp, vp, vp, vp]
    lib.specdec_build_tree_mask.restype = i32
    lib.specdec_profile_start.argtypes = [i32]
    lib.specdec_profile_start.restype = i32
    lib.specdec_profile_read.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int), i32]
    lib.specdec_profile_read.restype = i32
    lib.specdec_profile_stop.argtypes = []
    lib.specdec_profile_stop.restype = i32
    lib.specdec_version.argtypes = []
    lib.specdec_version.restype = ctypes.c_char_p
    lib.specdec_last_error.argtypes = []
    lib.specdec_last_error.restype = ctypes.c_char_p
    lib.specdec_set_test_hook.argtypes = [i32, i32]
    lib.specdec_set_test_hook.restype = i32
    lib.specdec_get_test_hook.argtypes = [i32]
    lib.specdec_get_test_hook.restype = i32
    _LIB = lib
    return lib


def _check(rc: int, what: str):
    if rc != OK:
        detail = ""
        if rc == ERR_CUDA:
            detail = ": " + load_library().specdec_last_error().decode(errors="replace")
        raise SpecdecError(f"{what}: {_ERR_NAMES.get(rc, rc)} (code {rc}){detail}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise ValueError(f"logits must be bfloat16 or float32, got {t.dtype}")


def _need(t: torch.Tensor, name: str, dtype, shape, device):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


_WORKSPACES: dict = {}


def _workspace(nbytes: int, device, stream_handle: int):
    """A device workspace per (device, stream); the library clears what it needs."""
    if nbytes == 0:
        return None, 0
    key = (device, stream_handle)
    ws = _WORKSPACES.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.zeros(max(nbytes, 1 << 16), dtype=torch.uint8, device=device)
        _WORKSPACES[key] = ws
    return ws, ws.numel()


def set_test_hook(hook: int, value: int) -> None:
    """Set one of the library's test hooks (HOOK_*; 0 restores the production behaviour)."""
    _check(load_library().specdec_set_test_hook(int(hook), int(value)), "specdec_set_test_hook")


def get_test_hook(hook: int) -> int:
    return int(load_library().specdec_get_test_hook(int(hook)))


class test_hooks:
    """Context manager: the given hooks set for the block, their previous values restored."""

    def __init__(self, **hooks):
        self.hooks = {globals()["HOOK_" + k.upper()]: int(v) for k, v in hooks.items()}
        self.saved = {}

    def __enter__(self):
        for h, v in self.hooks.items():
            self.saved[h] = get_test_hook(h)
            set_test_hook(h, v)
        return self

    def __exit__(self, *exc):
        for h, v in self.saved.items():
            set_test_hook(h, v)


def chain_workspace_bytes(B: int, gamma: int, V: int, dtype=torch.bfloat16) -> int:
    code = BF16 if dtype == torch.bfloat16 else F32
    return int(load_library().specdec_chain_workspace_bytes(B, gamma, V, code))


class _HostRoundTrip:
    """Copies host inputs to the device and device outputs back (argument marshalling).

    Every copy runs on the stream the library call runs on (the caller's `stream`, else the
    device's current stream), so that the inputs land before the kernels read them and the
    outputs are read after the kernels wrote them, whichever stream the caller chose."""

    def __init__(self, tensors, stream=None):
        self.on_host = tensors[0].device.type == "cpu"
        self.device = torch.device("cuda", torch.cuda.current_device()) if self.on_host else tensors[0].device
        self.stream = stream if stream is not None else (
            torch.cuda.current_stream(self.device) if self.on_host else None)
        # torch copies go to the current stream: switch only for a caller's other stream
        self.switch = self.on_host and stream is not None and stream != torch.cuda.current_stream(self.device)

    def _on_stream(self):
        return torch.cuda.stream(self.stream) if self.switch else contextlib.nullcontext()

    def to_device(self, t):
        if t is None or not self.on_host:
            return t
        with self._on_stream():
            return t.to(self.device, non_blocking=True)

    def to_device_all(self, *ts):
        if not self.on_host:
            return ts
        with self._on_stream():
            return tuple(None if t is None else t.to(self.device, non_blocking=True) for t in ts)

    def rows(self, t):
        """The logits and draft-probability rows of the chain calls: pinned host tensors stay
        on the host (the library reads the rows it needs over the host link), others are
        copied like every other input."""
        if t is None or not self.on_host or (t.is_pinned() and t.is_contiguous()):
            return t
        return self.to_device(t)

    def outputs(self, out):
        """The call's outputs (a tensor or a dict of tensors): on the host, for host inputs,
        copied on the call's stream and waited for once."""
        if not self.on_host:
            return out
        with self._on_stream():
            if isinstance(out, dict):
                res = {k: (None if v is None else v.to("cpu", non_blocking=True)) for k, v in out.items()}
            else:
                res = out.to("cpu", non_blocking=True)
        self.stream.synchronize()
        return res


def verify_chain(logits, draft_probs, draft_tokens, temperatures, uniforms, *, out=None,
                 with_p_draft: bool = True, stream=None) -> dict:
    """One round of chain verification per sequence (specdec_verify_chain).

    logits [B, g+1, V] bf16/fp32; draft_probs [B, g, V] fp32; draft_tokens [B, g] int32;
    temperatures [B] fp32; uniforms [B, g+1] fp32.  Returns a dict with tokens
    [B, g+1] int32 (-1 padded), num_accepted [B] int32, p_draft [B, g] fp32 (if
    requested) and status [B] int32.  Host tensors are copied to the current device and
    the results copied back, except pinned host logits and draft_probs: the library reads
    the rows the round needs from them in place, over the host link.
    """
    return _verify_round("specdec_verify_chain", "specdec_chain_workspace_bytes", logits, draft_probs,
                         draft_tokens, temperatures, uniforms, out, with_p_draft, stream, rows_on_host=True)


def verify_chain_varlen(logits, draft_probs, draft_tokens, temperatures, uniforms, gammas, *, out=None,
                        with_p_draft: bool = True, stream=None) -> dict:
    """Chain verification of the first gammas[b] drafts of each sequence
    (specdec_verify_chain_varlen); gammas [B] int32 in [0, g].  Results as verify_chain."""
    lib = load_library()
    rt = _HostRoundTrip([logits], stream)
    gammas = rt.to_device(gammas)
    B = logits.shape[0]
    _need(gammas, "gammas", torch.int32, (B,), gammas.device)

    class _Entry:  # the varlen call with the chain call's argument order
        def __call__(self, lg, code, q, d, T, u, B_, g, V, t, J, pd, st, ws, wsb, s_):
            return lib.specdec_verify_chain_varlen(lg, code, q, d, T, u, _ptr(gammas), B_, g, V, t, J, pd, st, ws,
                                                   wsb, s_)

    return _verify_round(_Entry(), "specdec_chain_workspace_bytes", logits, draft_probs, draft_tokens,
                         temperatures, uniforms, out, with_p_draft, stream, rows_on_host=True)


def verify_block(logits, draft_probs, draft_tokens, temperatures, uniforms, *, out=None,
                 with_p_draft: bool = True, stream=None) -> dict:
    """One round of block verification per sequence (specdec_verify_block): the draft is
    judged jointly.  Same arguments and results as verify_chain."""
    return _verify_round("specdec_verify_block", "specdec_block_workspace_bytes", logits, draft_probs,
                         draft_tokens, temperatures, uniforms, out, with_p_draft, stream)


def _verify_round(entry: str, ws_entry: str, logits, draft_probs, draft_tokens, temperatures, uniforms,
                  out, with_p_draft, stream, rows_on_host: bool = False) -> dict:
    lib = load_library()
    rt = _HostRoundTrip([logits], stream)
    rows = rt.rows if rows_on_host else rt.to_device
    logits, draft_probs = rows(logits), rows(draft_probs)
    draft_tokens, temperatures, uniforms = rt.to_device_all(draft_tokens, temperatures, uniforms)
    if logits.dim() != 3:
        raise ValueError("logits must be [B, g+1, V]")
    B, g1, V = logits.shape
    g = g1 - 1
    dev = rt.device
    code = _dtype_code(logits)
    _need(draft_probs, "draft_probs", torch.float32, (B, g, V), draft_probs.device if rt.on_host else dev)
    _need(draft_tokens, "draft_tokens", torch.int32, (B, g), dev)
    _need(temperatures, "temperatures", torch.float32, (B,), dev)
    _need(uniforms, "uniforms", torch.float32, (B, g1), dev)
    _need(logits, "logits", None, (B, g1, V), logits.device if rt.on_host else dev)
    if out is None:
        out = {
            "tokens": torch.empty(B, g1, dtype=torch.int32, device=dev),
            "num_accepted": torch.empty(B, dtype=torch.int32, device=dev),
            "status": torch.empty(B, dtype=torch.int32, device=dev),
        }
        if with_p_draft:
            out["p_draft"] = torch.empty(B, g, dtype=torch.float32, device=dev)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    if rows_on_host and logits.device.type == "cpu":
        # room for the device copy of each sequence's latest row (drawn rows are then not
        # read over the host link twice)
        ws_entry = "specdec_chain_host_workspace_bytes"
    ws, wsb = _workspace(int(getattr(lib, ws_entry)(B, g, V, code)), dev, s.cuda_stream)
    fn = getattr(lib, entry) if isinstance(entry, str) else entry

    def call(lg, qp):
        return fn(
            _ptr(lg), code, _ptr(qp), _ptr(draft_tokens), _ptr(temperatures),
            _ptr(uniforms), B, g, V, _ptr(out["tokens"]), _ptr(out["num_accepted"]),
            _ptr(out.get("p_draft")), _ptr(out.get("status")), _ptr(ws), wsb,
            ctypes.c_void_p(s.cuda_stream))

    rc = call(logits, draft_probs)
    if rc == ERR_UNSUPPORTED and rt.on_host and (logits.device.type == "cpu" or draft_probs.device.type == "cpu"):
        # rows the kernel cannot read in place (unaligned rows, sizes beyond the
        # left-to-right kernel): copy them like the other inputs
        rc = call(rt.to_device(logits), rt.to_device(draft_probs))
    _check(rc, entry if isinstance(entry, str) else "specdec_verify_chain_varlen")
    return rt.outputs(out)


def verify_greedy(logits, draft_tokens, *, out=None, stream=None) -> dict:
    """Greedy verification (specdec_verify_greedy): tokens, num_accepted, status."""
    lib = load_library()
    rt = _HostRoundTrip([logits], stream)
    logits, draft_tokens = rt.rows(logits), rt.to_device(draft_tokens)
    B, g1, V = logits.shape
    g = g1 - 1
    dev = rt.device
    code = _dtype_code(logits)
    _need(draft_tokens, "draft_tokens", torch.int32, (B, g), dev)
    _need(logits, "logits", None, (B, g1, V), logits.device if rt.on_host else dev)
    if out is None:
        out = {
            "tokens": torch.empty(B, g1, dtype=torch.int32, device=dev),
            "num_accepted": torch.empty(B, dtype=torch.int32, device=dev),
            "status": torch.empty(B, dtype=torch.int32, device=dev),
        }
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    ws, wsb = _workspace(int(lib.specdec_greedy_workspace_bytes(B, g, V, code)), dev, s.cuda_stream)
    def call(lg):
        return lib.specdec_verify_greedy(_ptr(lg), code, _ptr(draft_tokens), B, g, V,
                                         _ptr(out["tokens"]), _ptr(out["num_accepted"]),
                                         _ptr(out.get("status")), _ptr(ws), wsb,
                                         ctypes.c_void_p(s.cuda_stream))

    rc = call(logits)
    if rc == ERR_UNSUPPORTED and logits.device.type == "cpu":  # rows the kernel cannot read in place
        rc = call(rt.to_device(logits))
    _check(rc, "specdec_verify_greedy")
    return rt.outputs(out)


def verify_tree(logits, node_tokens, parents, temperatures, uniforms, max_depth: int, *,
                out=None, stream=None) -> dict:
    """Medusa tree walk (specdec_verify_tree): tokens [B, D+1], path [B, D],
    num_accepted [B], status [B]."""
    lib = load_library()
    rt = _HostRoundTrip([logits], stream)
    logits, node_tokens, parents, temperatures, uniforms = rt.to_device_all(
        logits, node_tokens, parents, temperatures, uniforms)
    B, n1, V = logits.shape
    N = n1 - 1
    D = int(max_depth)
    dev = logits.device
    code = _dtype_code(logits)
    _need(node_tokens, "node_tokens", torch.int32, (B, N), dev)
    _need(parents, "parents", torch.int32, (N,), dev)
    _need(temperatures, "temperatures", torch.float32, (B,), dev)
    _need(uniforms, "uniforms", torch.float32, (B, D + 1), dev)
    _need(logits, "logits", None, (B, n1, V), dev)
    if out is None:
        out = {
            "tokens": torch.empty(B, D + 1, dtype=torch.int32, device=dev),
            "path": torch.empty(B, D, dtype=torch.int32, device=dev),
            "num_accepted": torch.empty(B, dtype=torch.int32, device=dev),
            "status": torch.empty(B, dtype=torch.int32, device=dev),
        }
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    ws, wsb = _workspace(int(lib.specdec_tree_workspace_bytes(B, N, V, D, code)), dev, s.cuda_stream)
    rc = lib.specdec_verify_tree(_ptr(logits), code, _ptr(node_tokens), _ptr(parents),
                                 _ptr(temperatures), _ptr(uniforms), B, N, V, D,
                                 _ptr(out["tokens"]), _ptr(out["path"]), _ptr(out["num_accepted"]),
                                 _ptr(out.get("status")), _ptr(ws), wsb,
                                 ctypes.c_void_p(s.cuda_stream))
    _check(rc, "specdec_verify_tree")
    return rt.outputs(out)


def verify_tree_recursive(logits, draft_probs, node_tokens, parents, temperatures, uniforms, max_depth: int, *,
                          without_replacement: bool = False, out=None, stream=None) -> dict:
    """Sampled tree verification by recursive rejection (specdec_verify_tree_recursive).

    logits [B, N+1, V] bf16/fp32; draft_probs [B, N+1, V] fp32 (row 0: the root's children
    were drafted from it, row 1+i: node i's children); node_tokens [B, N] int32; parents
    [N] int32; temperatures [B]; uniforms [B, N+1] (slot 1+j tests node j, slot 0 the final
    draw).  without_replacement: every node's children were drawn without replacement
    (SPECDEC_TREE_WITHOUT_REPLACEMENT).  Returns tokens [B, D+1], path [B, D],
    num_accepted [B], status [B]."""
    lib = load_library()
    rt = _HostRoundTrip([logits], stream)
    logits, draft_probs, node_tokens, parents, temperatures, uniforms = rt.to_device_all(
        logits, draft_probs, node_tokens, parents, temperatures, uniforms)
    B, n1, V = logits.shape
    N = n1 - 1
    D = int(max_depth)
    dev = logits.device
    code = _dtype_code(logits)
    _need(draft_probs, "draft_probs", torch.float32, (B, n1, V), dev)
    _need(node_tokens, "node_tokens", torch.int32, (B, N), dev)
    _need(parents, "parents", torch.int32, (N,), dev)
    _need(temperatures, "temperatures", torch.float32, (B,), dev)
    _need(uniforms, "uniforms", torch.float32, (B, n1), dev)
    _need(logits, "logits", None, (B, n1, V), dev)
    if out is None:
        out = {
            "tokens": torch.empty(B, D + 1, dtype=torch.int32, device=dev),
            "path": torch.empty(B, D, dtype=torch.int32, device=dev),
            "num_accepted": torch.empty(B, dtype=torch.int32, device=dev),
            "status": torch.empty(B, dtype=torch.int32, device=dev),
        }
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    rc = lib.specdec_verify_tree_recursive(_ptr(logits), code, _ptr(draft_probs), _ptr(node_tokens), _ptr(parents),
                                           _ptr(temperatures), _ptr(uniforms), B, N, V, D,
                                           TREE_WITHOUT_REPLACEMENT if without_replacement else 0,
                                           _ptr(out["tokens"]), _ptr(out["path"]), _ptr(out["num_accepted"]),
                                           _ptr(out.get("status")), ctypes.c_void_p(s.cuda_stream))
    _check(rc, "specdec_verify_tree_recursive")
    return rt.outputs(out)


def verify_gumbel(logits, draft_tokens, temperatures, seed: int, *, out=None, stream=None) -> dict:
    """Gumbel-coupled verification (specdec_verify_gumbel): tokens [B, g+1], num_accepted
    [B], status [B].  The noise is Philox4x32-10 keyed by `seed` (0 <= seed < 2^64)."""
    lib = load_library()
    rt = _HostRoundTrip([logits], stream)
    logits, draft_tokens, temperatures = rt.to_device_all(logits, draft_tokens, temperatures)
    B, g1, V = logits.shape
    g = g1 - 1
    dev = logits.device
    code = _dtype_code(logits)
    _need(draft_tokens, "draft_tokens", torch.int32, (B, g), dev)
    _need(temperatures, "temperatures", torch.float32, (B,), dev)
    _need(logits, "logits", None, (B, g1, V), dev)
    if out is None:
        out = {"tokens": torch.empty(B, g1, dtype=torch.int32, device=dev),
               "num_accepted": torch.empty(B, dtype=torch.int32, device=dev),
               "status": torch.empty(B, dtype=torch.int32, device=dev)}
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    ws, wsb = _workspace(int(lib.specdec_gumbel_workspace_bytes(B, g)), dev, s.cuda_stream)
    rc = lib.specdec_verify_gumbel(_ptr(logits), code, _ptr(draft_tokens), _ptr(temperatures), int(seed), B, g, V,
                                   _ptr(out["tokens"]), _ptr(out["num_accepted"]), _ptr(out.get("status")),
                                   _ptr(ws), wsb, ctypes.c_void_p(s.cuda_stream))
    _check(rc, "specdec_verify_gumbel")
    return rt.outputs(out)


def gumbel_draft(draft_probs, seed: int, *, out=None, stream=None):
    """The drafter's shared-noise sampler (specdec_gumbel_draft): draft tokens [B, g]."""
    lib = load_library()
    rt = _HostRoundTrip([draft_probs], stream)
    draft_probs = rt.to_device(draft_probs)
    B, g, V = draft_probs.shape
    dev = draft_probs.device
    _need(draft_probs, "draft_probs", torch.float32, (B, g, V), dev)
    if out is None:
        out = torch.empty(B, g, dtype=torch.int32, device=dev)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    rc = lib.specdec_gumbel_draft(_ptr(draft_probs), int(seed), B, g, V, _ptr(out), ctypes.c_void_p(s.cuda_stream))
    _check(rc, "specdec_gumbel_draft")
    return rt.outputs(out)


def gumbel_noise(seed: int, B: int, rows: int, V: int, device=None, stream=None):
    """The shared Gumbel noise G [B, rows, V] fp32 (specdec_gumbel_noise)."""
    lib = load_library()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    out = torch.empty(B, rows, V, dtype=torch.float32, device=dev)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    _check(lib.specdec_gumbel_noise(int(seed), B, rows, V, _ptr(out), ctypes.c_void_p(s.cuda_stream)),
           "specdec_gumbel_noise")
    return out


def compact_kv(cache, prefix_len, path, num_accepted, *, block_table=None, stream=None) -> dict:
    """Accepted-branch KV compaction in place (specdec_compact_kv).

    cache: a device tensor [B, S, ...] (contiguous per sequence) or, with block_table
    [B, max_blocks] int32, a page pool [num_blocks, block_size, ...]; the trailing
    dimensions are one slot.  prefix_len [B], path [B, D], num_accepted [B] int32 (the tree
    verifier's outputs).  Returns new_len [B] and status [B]."""
    lib = load_library()
    if not cache.is_contiguous():
        raise ValueError("cache must be contiguous")
    dev = cache.device
    B = prefix_len.shape[0]
    D = path.shape[1]
    _need(prefix_len, "prefix_len", torch.int32, (B,), dev)
    _need(path, "path", torch.int32, (B, D), dev)
    _need(num_accepted, "num_accepted", torch.int32, (B,), dev)
    row = cache[0, 0].numel() * cache.element_size()
    slots = cache.shape[1]
    if block_table is not None:
        _need(block_table, "block_table", torch.int32, (B, block_table.shape[1]), dev)
        bs, mb, bstride, sstride, nslots = slots, block_table.shape[1], slots * row, 0, 0
    else:
        if cache.shape[0] != B:
            raise ValueError("cache must be [B, S, ...] without a block table")
        bs, mb, bstride, sstride, nslots = 0, 0, 0, slots * row, slots
    new_len = torch.empty(B, dtype=torch.int32, device=dev)
    status = torch.empty(B, dtype=torch.int32, device=dev)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    _check(lib.specdec_compact_kv(_ptr(cache), row, row, sstride, nslots, _ptr(block_table), bs, mb, bstride, B,
                                  _ptr(prefix_len), _ptr(path), D, _ptr(num_accepted), _ptr(new_len), _ptr(status),
                                  ctypes.c_void_p(s.cuda_stream)), "specdec_compact_kv")
    return {"new_len": new_len, "status": status}


def build_tree_mask(parents, prefix_len: int, *, stream=None) -> dict:
    """Tree-attention mask [N, P+N] uint8, position ids [N] int64, depth [N] int32 and a
    one-element status (specdec_build_tree_mask)."""
    lib = load_library()
    rt = _HostRoundTrip([parents], stream)
    parents = rt.to_device(parents)
    if parents.dim() != 1 or parents.dtype != torch.int32 or not parents.is_contiguous():
        raise ValueError("parents must be a contiguous int32 vector")
    N = parents.shape[0]
    dev = parents.device
    out = {
        "mask": torch.empty(N, prefix_len + N, dtype=torch.uint8, device=dev),
        "position_ids": torch.empty(N, dtype=torch.int64, device=dev),
        "depth": torch.empty(N, dtype=torch.int32, device=dev),
        "status": torch.empty(1, dtype=torch.int32, device=dev),
    }
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    rc = lib.specdec_build_tree_mask(_ptr(parents), N, int(prefix_len), _ptr(out["mask"]),
                                     _ptr(out["position_ids"]), _ptr(out["depth"]),
                                     _ptr(out["status"]), ctypes.c_void_p(s.cuda_stream))
    _check(rc, "specdec_build_tree_mask")
    return rt.outputs(out)


class KernelTimer:
    """Per-kernel CUDA-event timing of every library launch while active."""

    def __init__(self, max_launches: int = 4096):
        self.max_launches = max_launches

    def __enter__(self):
        _check(load_library().specdec_profile_start(self.max_launches), "specdec_profile_start")
        return self

    def read(self) -> dict:
        n = len(KERNEL_NAMES)
        ms = (ctypes.c_double * n)()
        cnt = (ctypes.c_int * n)()
        _check(load_library().specdec_profile_read(ms, cnt, n), "specdec_profile_read")
        return {KERNEL_NAMES[i]: (ms[i], cnt[i]) for i in range(n)}

    def __exit__(self, *exc):
        load_library().specdec_profile_stop()
        return False
