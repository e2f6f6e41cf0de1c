"""The C-ABI library builds, loads and exports every entry point declared in
include/ssdv.h; host-side validation answers without touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ssdv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ssd_[a-z_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_verification_draft_gb300 import build
    try:
        build.nvcc()
    except RuntimeError:
        pytest.skip("nvcc not available")
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ("ssd_verify", "ssd_verify_pipelined", "ssd_verify_noalloc", "ssd_verify_ragged",
                 "ssd_verify_ragged_pipelined",
                 "ssd_saguaro_prespec", "ssd_saguaro_workspace_bytes", "ssd_workspace_bytes",
                 "ssd_verify_saguaro", "ssd_cache_check", "ssd_verify_saguaro_draft", "ssd_verify_top_p",
                 "ssd_verify_top_p_workspace_bytes",
                 "ssd_workspace_init", "ssd_debug_rowstats", "ssd_debug_saguaro_stats",
                 "ssd_debug_uniforms", "ssd_read_status", "ssd_status_str", "ssd_last_error"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"libssdv.so does not export {name}"


def test_host_validation_without_gpu(lib):
    from speculative_decoding_verification_draft_gb300 import ssdv
    L = ssdv._declare(lib)
    assert L.ssd_workspace_bytes(64, 4) >= 16 + 4 * 64 + 2 * 4 * 64 * 5
    assert L.ssd_workspace_bytes(0, 4) == 0
    # temperature rejected first
    assert L.ssd_verify(None, None, 0, None, 1, 1, 8, -1.0, 0, None, None, None, 0, None) == 6
    assert L.ssd_verify(None, None, 0, None, 1, 1, 8, float("nan"), 0, None, None, None, 0, None) == 6
    assert L.ssd_verify(None, None, 0, None, 1, 1, 8, 1e-9, 0, None, None, None, 0, None) == 6
    # unknown dtype, NULL pointers
    assert L.ssd_verify(None, None, 7, None, 1, 1, 8, 1.0, 0, None, None, None, 0, None) == 3
    assert L.ssd_verify(None, None, 0, None, 1, 1, 8, 1.0, 0, None, None, None, 0, None) == 1
    assert b"NULL" in L.ssd_last_error()
    # shape checks run before any device query
    p = ctypes.c_void_p(16)
    assert L.ssd_verify(p, p, 0, p, 0, 1, 8, 1.0, 0, p, p, p, 1 << 20, None) == 2
    # one past each declared maximum: gamma 32 (SSD_MAX_GAMMA 31), V 2^19 + 1 (SSD_MAX_V)
    assert L.ssd_verify(p, p, 0, p, 1, 32, 8, 1.0, 0, p, p, p, 1 << 20, None) == 2
    assert L.ssd_verify(p, p, 0, p, 1, 1, (1 << 19) + 1, 1.0, 0, p, p, p, 1 << 20, None) == 2
    assert L.ssd_saguaro_prespec(p, p, 0, 1, 32, 8, 3, 0, 1.0, 0, p, p, p, 1 << 20, None) == 2
    assert L.ssd_saguaro_prespec(p, p, 0, 1, 1, (1 << 19) + 1, 3, 0, 1.0, 0, p, p, p, 1 << 20, None) == 2
    assert L.ssd_verify(p, p, 0, p, 1, 33, 8, 1.0, 0, p, p, p, 1 << 20, None) == 2
    # misaligned bf16 pointer, small workspace
    odd = ctypes.c_void_p(17)
    assert L.ssd_verify(odd, p, 0, p, 1, 1, 8, 1.0, 0, p, p, p, 1 << 20, None) == 4
    assert L.ssd_verify(p, p, 0, p, 4, 2, 8, 1.0, 0, p, p, p, 8, None) == 9
    # Saguaro: k and temperature
    assert L.ssd_saguaro_prespec(p, p, 0, 1, 1, 8, 9, 0, 1.0, 0, p, p, p, 1 << 20, None) == 2
    assert L.ssd_saguaro_prespec(p, p, 0, 1, 1, 8, 3, 0, 0.0, 0, p, p, p, 1 << 20, None) == 6
    assert L.ssd_saguaro_prespec(p, p, 0, 1, 1, 8, 3, 0, 1.0, 0, p, p, None, 1 << 20, None) == 1
    assert L.ssd_saguaro_prespec(p, p, 0, 4, 2, 8, 3, 0, 1.0, 0, p, p, p, 8, None) == 9
    assert L.ssd_saguaro_prespec(p, p, 0, 1, 1, 8, 3, 2, 1.0, 0, p, p, p, 1 << 20, None) == 2  # unknown source
    # fused call: greedy rejected; cache check: needs an output, k in range
    assert L.ssd_verify_saguaro(p, p, 0, p, 1, 1, 8, 3, 0, 0.0, 0, p, p, p, p, None, None, p, 1 << 20, None) == 6
    assert L.ssd_verify_saguaro(p, p, 0, p, 1, 1, 8, 3, 0, 1.0, 0, None, p, p, p, None, None, p, 1 << 20,
                                None) == 1
    assert L.ssd_cache_check(p, p, p, 4, 2, 3, None, None, None) == 1
    # top-p: top_p in (0, 1]; its workspace is larger than plain verification's
    assert L.ssd_verify_top_p(p, p, 0, p, 1, 1, 8, 1.0, 0.0, 0, p, p, p, 1 << 20, None) == 2
    assert L.ssd_verify_top_p(p, p, 0, p, 1, 1, 8, 1.0, 1.5, 0, p, p, p, 1 << 20, None) == 2
    assert L.ssd_verify_top_p_workspace_bytes(8, 4) > L.ssd_workspace_bytes(8, 4)
    # verification under Saguaro sampling: greedy rejected, workspace sized by V
    assert L.ssd_verify_saguaro_draft(p, p, 0, p, 1, 1, 8, 0.0, 0, p, p, p, 1 << 20, None) == 6
    assert L.ssd_verify_saguaro_draft(p, p, 0, p, 4, 2, 8, 1.0, 0, p, p, p, 8, None) == 9
    assert L.ssd_cache_check(p, p, p, 4, 2, 9, p, None, None) == 2
    # ragged calls, plain and pipelined: the per-request arrays are required,
    # then the shape and the workspace are checked as for ssd_verify
    for fn in (L.ssd_verify_ragged, L.ssd_verify_ragged_pipelined):
        assert fn(p, p, 0, p, 1, 1, 8, None, p, 0, p, p, p, 1 << 20, None) == 1
        assert fn(p, p, 0, p, 1, 1, 8, p, None, 0, p, p, p, 1 << 20, None) == 1
        assert fn(p, p, 0, p, 0, 1, 8, p, p, 0, p, p, p, 1 << 20, None) == 2
        assert fn(p, p, 0, p, 4, 2, 8, p, p, 0, p, p, p, 8, None) == 9
    # Saguaro workspace: zero for a bad shape, grows with the vocabulary
    assert L.ssd_saguaro_workspace_bytes(0, 1, 8) == 0
    assert L.ssd_saguaro_workspace_bytes(4, 2, 1 << 17) > L.ssd_saguaro_workspace_bytes(4, 2, 1 << 10)
    for code in range(12):
        assert L.ssd_status_str(code).startswith(b"SSD_")


def test_binding_has_no_host_fallback(monkeypatch):
    """The Python binding only marshals device tensors into the C ABI: host
    tensors are refused before any call, and a missing library is an error,
    not a switch to some other implementation."""
    import torch
    from speculative_decoding_verification_draft_gb300 import ssdv
    t = torch.zeros(2, 3, 16, dtype=torch.bfloat16)
    d = torch.zeros(2, 2, 16, dtype=torch.bfloat16)
    k = torch.zeros(2, 2, dtype=torch.int32)
    ws = torch.zeros(1 << 16, dtype=torch.uint8)
    with pytest.raises(ValueError, match="CUDA device"):
        ssdv.verify(t, d, k, 1.0, 0, workspace=ws)
    with pytest.raises(ValueError, match="CUDA device"):
        ssdv.verify_ragged(t, d, k, torch.full((2,), 2, dtype=torch.int32), torch.ones(2), 0, workspace=ws,
                           pipelined=True)
    monkeypatch.setattr(ssdv, "_lib", None)
    monkeypatch.setattr(ssdv, "LIBRARY", os.path.join(ROOT, "no_such_dir", "libssdv.so"))
    with pytest.raises(RuntimeError, match="missing"):
        ssdv.lib()
