"""C-ABI checks that need no GPU: the library builds, loads, exports every declared
symbol, and rejects invalid arguments on the host before touching the device."""
import ctypes
import re
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]
HEADER = ROOT / "include" / "specdec.h"


def declared_functions():
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(specdec_[A-Za-z0-9_]+)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_four_verification_calls():
    names = declared_functions()
    for fn in ("specdec_verify_chain", "specdec_verify_greedy", "specdec_verify_tree",
               "specdec_build_tree_mask", "specdec_verify_block", "specdec_verify_tree_recursive",
               "specdec_verify_gumbel", "specdec_gumbel_draft", "specdec_gumbel_noise",
               "specdec_verify_chain_varlen", "specdec_compact_kv", "specdec_gumbel_workspace_bytes"):
        assert fn in names


def test_library_exports_every_declared_symbol(built_library):
    lib = ctypes.CDLL(str(built_library))
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_loads_and_reports_version(built_library):
    import speculative_decoding_token_temperature_gb300 as sd
    lib = sd.load_library()
    assert lib.specdec_version().decode().count(".") == 2


def test_workspace_sizes(built_library):
    import speculative_decoding_token_temperature_gb300 as sd
    lib = sd.load_library()
    a = lib.specdec_chain_workspace_bytes(256, 7, 128256, sd.BF16)
    b = lib.specdec_chain_workspace_bytes(512, 8, 152064, sd.F32)
    assert 0 < a < b
    assert a % 256 == 0
    assert lib.specdec_chain_workspace_bytes(0, 7, 10, sd.BF16) == 0
    assert lib.specdec_chain_workspace_bytes(1, 7, 10, 9) == 0
    assert lib.specdec_greedy_workspace_bytes(4, 3, 100, sd.F32) == lib.specdec_chain_workspace_bytes(4, 3, 100, sd.F32)
    # block verification keeps every row's residual masses: more than the chain's
    blk = lib.specdec_block_workspace_bytes(256, 7, 128256, sd.BF16)
    assert blk > a and blk % 256 == 0
    assert lib.specdec_block_workspace_bytes(0, 7, 10, sd.BF16) == 0
    assert lib.specdec_block_workspace_bytes(1, 7, 10, 9) == 0
    # host-resident logits: room for one device copy of a row per sequence on top
    for B_, g_, V_, code, es in ((256, 7, 128256, sd.BF16, 2), (3, 2, 1000, sd.F32, 4), (1, 1, 8, sd.BF16, 2)):
        base = lib.specdec_chain_workspace_bytes(B_, g_, V_, code)
        extra = -(-(B_ * V_ * es) // 256) * 256
        assert lib.specdec_chain_host_workspace_bytes(B_, g_, V_, code) == base + extra
    assert lib.specdec_chain_host_workspace_bytes(0, 7, 10, sd.BF16) == 0
    assert lib.specdec_chain_host_workspace_bytes(1, 7, 10, 9) == 0


def _fake(n=64):
    """256-byte aligned host addresses that are never dereferenced: validation rejects
    the call before any use."""
    buf = (ctypes.c_byte * (n + 256))()
    addr = ctypes.addressof(buf)
    return ctypes.c_void_p((addr + 255) // 256 * 256), buf


def test_host_validation_rejects_before_launch(built_library):
    import speculative_decoding_token_temperature_gb300 as sd
    lib = sd.load_library()
    p, keep = _fake()
    ws, keep2 = _fake(1 << 12)
    # null logits
    assert lib.specdec_verify_chain(None, sd.BF16, p, p, p, p, 1, 1, 8, p, p, None, None, ws, 4096, None) == sd.ERR_INVALID_ARG
    # bad dtype
    assert lib.specdec_verify_chain(p, 7, p, p, p, p, 1, 1, 8, p, p, None, None, ws, 4096, None) == sd.ERR_INVALID_ARG
    # non-positive sizes
    for B, g, V in [(0, 1, 8), (1, 0, 8), (1, 1, 0), (-3, 1, 8)]:
        assert lib.specdec_verify_chain(p, sd.BF16, p, p, p, p, B, g, V, p, p, None, None, ws, 4096, None) == sd.ERR_INVALID_ARG
    # missing q / temperatures / uniforms on the sampling call
    assert lib.specdec_verify_chain(p, sd.BF16, None, p, p, p, 1, 1, 8, p, p, None, None, ws, 4096, None) == sd.ERR_INVALID_ARG
    # workspace too small, null, or misaligned
    assert lib.specdec_verify_chain(p, sd.BF16, p, p, p, p, 1, 1, 8, p, p, None, None, ws, 1, None) == sd.ERR_WORKSPACE
    assert lib.specdec_verify_chain(p, sd.BF16, p, p, p, p, 1, 1, 8, p, p, None, None, None, 4096, None) == sd.ERR_INVALID_ARG
    mis = ctypes.c_void_p(ws.value + 8)
    assert lib.specdec_verify_chain(p, sd.BF16, p, p, p, p, 1, 1, 8, p, p, None, None, mis, 4000, None) == sd.ERR_INVALID_ARG
    # too many drafts for one decision CTA
    assert lib.specdec_verify_chain(p, sd.BF16, p, p, p, p, 1, 300, 8, p, p, None, None, ws, 4096, None) == sd.ERR_UNSUPPORTED
    # greedy: null drafts
    assert lib.specdec_verify_greedy(p, sd.F32, None, 1, 1, 8, p, p, None, ws, 4096, None) == sd.ERR_INVALID_ARG
    # tree: bad depth, null outputs
    assert lib.specdec_verify_tree(p, sd.BF16, p, p, p, p, 1, 2, 8, 0, p, p, p, None, None, 0, None) == sd.ERR_INVALID_ARG
    assert lib.specdec_verify_tree(p, sd.BF16, p, p, p, p, 1, 2, 8, 100, p, p, p, None, None, 0, None) == sd.ERR_UNSUPPORTED
    assert lib.specdec_verify_tree(p, sd.BF16, p, p, p, p, 1, 2, 8, 2, None, p, p, None, None, 0, None) == sd.ERR_INVALID_ARG
    # block: null q, unaligned rows (V = 4 bf16 is 8 bytes), too many drafts, small workspace
    assert lib.specdec_verify_block(p, sd.BF16, None, p, p, p, 1, 1, 8, p, p, None, None, ws, 4096, None) == sd.ERR_INVALID_ARG
    assert lib.specdec_verify_block(p, sd.BF16, p, p, p, None, 1, 1, 8, p, p, None, None, ws, 4096, None) == sd.ERR_INVALID_ARG
    assert lib.specdec_verify_block(p, sd.BF16, p, p, p, p, 1, 1, 4, p, p, None, None, ws, 4096, None) == sd.ERR_UNSUPPORTED
    assert lib.specdec_verify_block(p, sd.BF16, p, p, p, p, 1, 32, 8, p, p, None, None, ws, 4096, None) == sd.ERR_UNSUPPORTED
    assert lib.specdec_verify_block(p, sd.BF16, p, p, p, p, 1, 1, 8, p, p, None, None, ws, 1, None) == sd.ERR_WORKSPACE
    assert lib.specdec_verify_block(p, sd.BF16, p, p, p, p, 0, 1, 8, p, p, None, None, ws, 4096, None) == sd.ERR_INVALID_ARG
    # recursive-rejection tree walk: null q, bad depth
    assert lib.specdec_verify_tree_recursive(p, sd.BF16, None, p, p, p, p, 1, 2, 8, 2, 0, p, p, p, None, None) == sd.ERR_INVALID_ARG
    assert lib.specdec_verify_tree_recursive(p, sd.BF16, p, p, p, p, p, 1, 2, 8, 0, 0, p, p, p, None, None) == sd.ERR_INVALID_ARG
    assert lib.specdec_verify_tree_recursive(p, sd.BF16, p, p, p, p, p, 1, 2, 8, 65, 0, p, p, p, None, None) == sd.ERR_UNSUPPORTED
    assert lib.specdec_verify_tree_recursive(p, 5, p, p, p, p, p, 1, 2, 8, 2, 0, p, p, p, None, None) == sd.ERR_INVALID_ARG
    # flag bits other than SPECDEC_TREE_WITHOUT_REPLACEMENT
    assert lib.specdec_verify_tree_recursive(p, sd.BF16, p, p, p, p, p, 1, 2, 8, 2, 2, p, p, p, None, None) == sd.ERR_INVALID_ARG
    # per-sequence draft counts: null counts; unaligned rows (V = 4 bf16) are refused
    assert lib.specdec_verify_chain_varlen(p, sd.BF16, p, p, p, p, None, 1, 1, 8, p, p, None, None, ws, 4096, None) == sd.ERR_INVALID_ARG
    assert lib.specdec_verify_chain_varlen(p, sd.BF16, p, p, p, p, p, 1, 1, 4, p, p, None, None, ws, 4096, None) == sd.ERR_UNSUPPORTED
    # KV compaction: null cache, bad sizes, a paged layout without a block size
    assert lib.specdec_compact_kv(None, 16, 16, 160, 10, None, 0, 0, 0, 1, p, p, 2, p, None, None, None) == sd.ERR_INVALID_ARG
    assert lib.specdec_compact_kv(p, 0, 16, 160, 10, None, 0, 0, 0, 1, p, p, 2, p, None, None, None) == sd.ERR_INVALID_ARG
    assert lib.specdec_compact_kv(p, 16, 16, 0, 10, p, 0, 4, 64, 1, p, p, 2, p, None, None, None) == sd.ERR_INVALID_ARG
    # Gumbel coupling: null drafts, bad sizes, too many rows per sequence
    assert lib.specdec_verify_gumbel(p, sd.BF16, None, p, 1, 1, 1, 8, p, p, None, ws, 4096, None) == sd.ERR_INVALID_ARG
    assert lib.specdec_verify_gumbel(p, sd.BF16, p, p, 1, 0, 1, 8, p, p, None, ws, 4096, None) == sd.ERR_INVALID_ARG
    assert lib.specdec_verify_gumbel(p, sd.BF16, p, p, 1, 1, 600, 8, p, p, None, ws, 4096, None) == sd.ERR_UNSUPPORTED
    assert lib.specdec_verify_gumbel(p, sd.BF16, p, p, 1, 64, 1, 8, p, p, None, ws, 16, None) == sd.ERR_WORKSPACE
    assert lib.specdec_gumbel_workspace_bytes(256, 7) > 0 and lib.specdec_gumbel_workspace_bytes(0, 7) == 0
    assert lib.specdec_gumbel_draft(None, 1, 1, 1, 8, p, None) == sd.ERR_INVALID_ARG
    assert lib.specdec_gumbel_draft(p, 1, 1, 1, 0, p, None) == sd.ERR_INVALID_ARG
    assert lib.specdec_gumbel_noise(1, 1, 1, 8, None, None) == sd.ERR_INVALID_ARG
    assert lib.specdec_gumbel_noise(1, 0, 1, 8, p, None) == sd.ERR_INVALID_ARG
    # mask
    assert lib.specdec_build_tree_mask(None, 4, 2, p, p, None, p, None) == sd.ERR_INVALID_ARG
    assert lib.specdec_build_tree_mask(p, 0, 2, p, p, None, p, None) == sd.ERR_INVALID_ARG
    assert lib.specdec_build_tree_mask(p, 4, -1, p, p, None, p, None) == sd.ERR_INVALID_ARG
    del keep, keep2


def test_binding_marshalling_errors_without_gpu(built_library):
    import torch
    import speculative_decoding_token_temperature_gb300 as sd
    with pytest.raises(ValueError):
        sd._dtype_code(torch.zeros(2, dtype=torch.float16))
    t = torch.zeros(2, 3)
    with pytest.raises(ValueError):
        sd._need(t, "x", torch.float32, (3, 2), t.device)
    with pytest.raises(ValueError):
        sd._need(t.t(), "x", torch.float32, (3, 2), t.device)


def test_test_hooks_are_validated_and_default_to_production(built_library):
    import speculative_decoding_token_temperature_gb300 as sd
    lib = sd.load_library()
    for h in range(5):
        assert lib.specdec_get_test_hook(h) == 0
    assert lib.specdec_set_test_hook(99, 1) == sd.ERR_INVALID_ARG
    assert lib.specdec_set_test_hook(-1, 0) == sd.ERR_INVALID_ARG
    assert lib.specdec_set_test_hook(sd.HOOK_TREE_CLUSTER, 3) == sd.ERR_INVALID_ARG
    assert lib.specdec_set_test_hook(sd.HOOK_CHAIN_ALL_ROWS, 2) == sd.ERR_INVALID_ARG
    assert lib.specdec_set_test_hook(sd.HOOK_QUEUE_WAIT_US, -5) == sd.ERR_INVALID_ARG
    with sd.test_hooks(tree_cluster=4, queue_wait_us=250):
        assert lib.specdec_get_test_hook(sd.HOOK_TREE_CLUSTER) == 4
        assert lib.specdec_get_test_hook(sd.HOOK_QUEUE_WAIT_US) == 250
    assert lib.specdec_get_test_hook(sd.HOOK_TREE_CLUSTER) == 0
    assert lib.specdec_get_test_hook(sd.HOOK_QUEUE_WAIT_US) == 0


def test_header_compiles_as_c_and_cpp(tmp_path):
    """include/specdec.h is plain C: a C99 and a C++17 translation unit that include it and
    name every entry point compile without a warning (no GPU, no CUDA headers needed)."""
    import re
    import shutil
    import subprocess
    hdr = ROOT / "include" / "specdec.h"
    names = sorted(set(re.findall(r"^(?:int|size_t|const char\s*\*)\s*(specdec_\w+)\(", hdr.read_text(), re.M)))
    assert len(names) > 20, names
    body = '#include "specdec.h"\ntypedef void (*fn_t)(void);\nint main(void) {\n  fn_t p[] = {'
    body += ", ".join(f"(fn_t){n}" for n in names) + "};\n  return p[0] == 0;\n}\n"
    for compiler, flags, suffix in (("gcc", ["-std=c99", "-pedantic"], ".c"), ("g++", ["-std=c++17"], ".cpp")):
        if shutil.which(compiler) is None:
            pytest.skip(f"{compiler} not found")
        src = tmp_path / ("probe" + suffix)
        src.write_text(body)
        r = subprocess.run([compiler, *flags, "-Wall", "-Wextra", "-Werror", f"-I{ROOT / 'include'}", "-c", str(src),
                            "-o", str(tmp_path / "probe.o")], capture_output=True, text=True)
        assert r.returncode == 0, (compiler, r.stderr[-2000:])
