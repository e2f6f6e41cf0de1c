"""Thin ctypes binding of libssdv (C ABI in ``include/ssdv.h``).

Argument marshalling only: every function checks tensor dtypes, shapes and
devices, passes raw device pointers and the current CUDA stream to the
library, and turns a non-zero status into ``SsdError``.  All computation runs
in the library's CUDA kernels; there is no CPU fallback.  If ``libssdv.so`` is
missing the first call raises -- build it with ``build.build()`` (or
``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.path.join(PKG, "libssdv.so")

SSD_BF16, SSD_F32 = 0, 1
NSTAT_VERIFY = 10
NSTAT_SAGUARO = 10
MAX_TOPK = 8

STATUS_NAMES = {
    0: "SSD_OK", 1: "SSD_ERR_NULL", 2: "SSD_ERR_SHAPE", 3: "SSD_ERR_DTYPE", 4: "SSD_ERR_ALIGN",
    5: "SSD_ERR_TOKEN_RANGE", 6: "SSD_ERR_TEMPERATURE", 7: "SSD_ERR_CUDA", 8: "SSD_ERR_UNSUPPORTED",
    9: "SSD_ERR_WORKSPACE", 10: "SSD_ERR_GAMMA", 11: "SSD_ERR_DRAW",
}


class SsdError(RuntimeError):
    def __init__(self, status: int, detail: str):
        self.status = status
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {detail}")


_lock = threading.Lock()
_lib = None


def _declare(lib):
    P, I, U64, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_float, ctypes.c_size_t
    lib.ssd_workspace_bytes.argtypes = [I, I]
    lib.ssd_workspace_bytes.restype = SZ
    lib.ssd_workspace_init.argtypes = [P, SZ, P]
    lib.ssd_verify.argtypes = [P, P, I, P, I, I, I, F, U64, P, P, P, SZ, P]
    lib.ssd_verify_ragged.argtypes = [P, P, I, P, I, I, I, P, P, U64, P, P, P, SZ, P]
    lib.ssd_verify_ragged_pipelined.argtypes = [P, P, I, P, I, I, I, P, P, U64, P, P, P, SZ, P]
    lib.ssd_verify_noalloc.argtypes = [P, P, I, P, I, I, I, F, U64, P, P, P]
    lib.ssd_verify_pipelined.argtypes = [P, P, I, P, I, I, I, F, U64, P, P, P, SZ, P]
    lib.ssd_saguaro_prespec.argtypes = [P, P, I, I, I, I, I, I, F, U64, P, P, P, SZ, P]
    lib.ssd_saguaro_workspace_bytes.argtypes = [I, I, I]
    lib.ssd_saguaro_workspace_bytes.restype = SZ
    lib.ssd_debug_rowstats.argtypes = [P, P, I, P, I, I, I, F, U64, P, P, P, P, SZ, P]
    lib.ssd_debug_saguaro_stats.argtypes = [P, P, I, I, I, I, I, I, F, U64, P, P, P, P, SZ, P]
    lib.ssd_verify_saguaro.argtypes = [P, P, I, P, I, I, I, I, I, F, U64, P, P, P, P, P, P, P, SZ, P]
    lib.ssd_cache_check.argtypes = [P, P, P, I, I, I, P, P, P]
    lib.ssd_verify_saguaro_draft.argtypes = [P, P, I, P, I, I, I, F, U64, P, P, P, SZ, P]
    lib.ssd_verify_top_p.argtypes = [P, P, I, P, I, I, I, F, F, U64, P, P, P, SZ, P]
    lib.ssd_verify_top_p_workspace_bytes.argtypes = [I, I]
    lib.ssd_verify_top_p_workspace_bytes.restype = SZ
    lib.ssd_read_status.argtypes = [P, SZ, P, P]
    lib.ssd_debug_uniforms.argtypes = [U64, I, I, P, P]
    lib.ssd_status_str.argtypes = [I]
    lib.ssd_status_str.restype = ctypes.c_char_p
    lib.ssd_last_error.argtypes = []
    lib.ssd_last_error.restype = ctypes.c_char_p
    for name in ("ssd_workspace_init", "ssd_verify", "ssd_verify_noalloc", "ssd_verify_pipelined",
                 "ssd_verify_ragged", "ssd_verify_ragged_pipelined", "ssd_saguaro_prespec", "ssd_debug_rowstats",
                 "ssd_debug_saguaro_stats", "ssd_read_status",
                 "ssd_verify_saguaro", "ssd_cache_check", "ssd_verify_saguaro_draft", "ssd_verify_top_p",
                 "ssd_debug_uniforms"):
        getattr(lib, name).restype = I
    return lib


def lib():
    """The loaded CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIBRARY):
                raise RuntimeError(f"{LIBRARY} is missing: build the CUDA library first "
                                   "(speculative_decoding_verification_draft_gb300.build.build())")
            _lib = _declare(ctypes.CDLL(LIBRARY))
    return _lib


def _check(status: int):
    if status != 0:
        raise SsdError(status, lib().ssd_last_error().decode())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SSD_BF16
    if t.dtype == torch.float32:
        return SSD_F32
    raise TypeError(f"logits must be bfloat16 or float32, got {t.dtype}")


def _dev(t: torch.Tensor, name: str, dtype=None) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


TOPK_SOURCES = {"residual": 0, "draft": 1}


def _source(source: str) -> int:
    if source not in TOPK_SOURCES:
        raise ValueError(f"top-k source must be one of {sorted(TOPK_SOURCES)}, got {source!r}")
    return TOPK_SOURCES[source]


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


_ws_cache = {}


def workspace_bytes(B: int, gamma_max: int) -> int:
    return int(lib().ssd_workspace_bytes(B, gamma_max))


def make_workspace(B: int, gamma_max: int, device=None) -> torch.Tensor:
    """A zeroed device workspace for batches of up to B requests / gamma_max."""
    n = workspace_bytes(B, gamma_max)
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def _ws_key(device):
    device = torch.device(device if device is not None else "cuda")
    index = device.index if device.index is not None else torch.cuda.current_device()
    return (index, torch.cuda.current_stream(index).cuda_stream)


def _workspace(B: int, gmax: int, device, given: Optional[torch.Tensor]):
    if given is not None:
        return given
    key = _ws_key(device)
    need = workspace_bytes(B, gmax)
    ws = _ws_cache.get(key)
    if ws is None or ws.numel() < need:
        ws = torch.zeros(max(need, 1 << 16), dtype=torch.uint8, device=device)
        _ws_cache[key] = ws
    return ws


_sag_ws_cache = {}


def saguaro_workspace_bytes(B: int, gamma: int, V: int) -> int:
    return int(lib().ssd_saguaro_workspace_bytes(B, gamma, V))


def make_saguaro_workspace(B: int, gamma: int, V: int, device=None) -> torch.Tensor:
    """A zeroed device workspace for Saguaro calls of up to B requests, gamma, V."""
    n = saguaro_workspace_bytes(B, gamma, V)
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def _saguaro_workspace(B: int, g: int, V: int, device, given: Optional[torch.Tensor]):
    # kept apart from the verification workspaces: a pipelined verification
    # call may write its workspace while the previous kernel still runs
    if given is not None:
        return given
    key = _ws_key(device)
    need = saguaro_workspace_bytes(B, g, V)
    ws = _sag_ws_cache.get(key)
    if ws is None or ws.numel() < need:
        ws = torch.zeros(max(need, 1 << 16), dtype=torch.uint8, device=device)
        _sag_ws_cache[key] = ws
    return ws


def verify(target: torch.Tensor, draft: Optional[torch.Tensor], draft_tokens: torch.Tensor,
           temperature: float, seed: int, out_tokens: Optional[torch.Tensor] = None,
           n_accepted: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
           stream=None):
    """ssd_verify: target [B, g+1, V], draft [B, g, V], draft_tokens [B, g] int32.

    Returns (out_tokens [B, g+1] int32, n_accepted [B] int32)."""
    B, W, V = target.shape
    g = W - 1
    dev = target.device
    if out_tokens is None:
        out_tokens = torch.empty(B, W, dtype=torch.int32, device=dev)
    if n_accepted is None:
        n_accepted = torch.empty(B, dtype=torch.int32, device=dev)
    ws = _workspace(B, g, dev, workspace)
    dptr = _dev(draft, "draft_logits", target.dtype) if draft is not None else None
    if draft is not None and tuple(draft.shape) != (B, g, V):
        raise ValueError("draft_logits must be [B, gamma, V]")
    if tuple(draft_tokens.shape) != (B, g):
        raise ValueError("draft_tokens must be [B, gamma]")
    _check(lib().ssd_verify(_dev(target, "target_logits"), dptr, _dtype_code(target),
                            _dev(draft_tokens, "draft_tokens", torch.int32), B, g, V, float(temperature),
                            int(seed) & ((1 << 64) - 1), _dev(out_tokens, "out_tokens", torch.int32),
                            _dev(n_accepted, "n_accepted", torch.int32), _dev(ws, "workspace"),
                            ws.numel(), _stream(stream)))
    return out_tokens, n_accepted


def verify_pipelined(target: torch.Tensor, draft: Optional[torch.Tensor], draft_tokens: torch.Tensor,
                     temperature: float, seed: int, out_tokens: Optional[torch.Tensor] = None,
                     n_accepted: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                     stream=None):
    """ssd_verify_pipelined: ssd_verify for a chain of calls whose inputs were
    complete before the previous verification call on the stream completed."""
    B, W, V = target.shape
    g = W - 1
    dev = target.device
    if out_tokens is None:
        out_tokens = torch.empty(B, W, dtype=torch.int32, device=dev)
    if n_accepted is None:
        n_accepted = torch.empty(B, dtype=torch.int32, device=dev)
    ws = _workspace(B, g, dev, workspace)
    dptr = _dev(draft, "draft_logits", target.dtype) if draft is not None else None
    if draft is not None and tuple(draft.shape) != (B, g, V):
        raise ValueError("draft_logits must be [B, gamma, V]")
    if tuple(draft_tokens.shape) != (B, g):
        raise ValueError("draft_tokens must be [B, gamma]")
    _check(lib().ssd_verify_pipelined(_dev(target, "target_logits"), dptr, _dtype_code(target),
                                      _dev(draft_tokens, "draft_tokens", torch.int32), B, g, V, float(temperature),
                                      int(seed) & ((1 << 64) - 1), _dev(out_tokens, "out_tokens", torch.int32),
                                      _dev(n_accepted, "n_accepted", torch.int32), _dev(ws, "workspace"),
                                      ws.numel(), _stream(stream)))
    return out_tokens, n_accepted


def verify_noalloc(target: torch.Tensor, draft: Optional[torch.Tensor], draft_tokens: torch.Tensor,
                   temperature: float, seed: int, out_tokens: torch.Tensor, n_accepted: torch.Tensor,
                   stream=None):
    """ssd_verify_noalloc: ssd_verify on the library's fixed device scratch.

    The caller passes the outputs (out_tokens [B, g+1], n_accepted [B] int32),
    so neither this wrapper nor the library allocates device memory."""
    B, W, V = target.shape
    g = W - 1
    dptr = _dev(draft, "draft_logits", target.dtype) if draft is not None else None
    if draft is not None and tuple(draft.shape) != (B, g, V):
        raise ValueError("draft_logits must be [B, gamma, V]")
    if tuple(draft_tokens.shape) != (B, g):
        raise ValueError("draft_tokens must be [B, gamma]")
    if tuple(out_tokens.shape) != (B, W) or tuple(n_accepted.shape) != (B,):
        raise ValueError("out_tokens must be [B, gamma+1] and n_accepted [B]")
    _check(lib().ssd_verify_noalloc(_dev(target, "target_logits"), dptr, _dtype_code(target),
                                    _dev(draft_tokens, "draft_tokens", torch.int32), B, g, V, float(temperature),
                                    int(seed) & ((1 << 64) - 1), _dev(out_tokens, "out_tokens", torch.int32),
                                    _dev(n_accepted, "n_accepted", torch.int32), _stream(stream)))
    return out_tokens, n_accepted


def verify_ragged(target: torch.Tensor, draft: torch.Tensor, draft_tokens: torch.Tensor,
                  gamma: torch.Tensor, temperature: torch.Tensor, seed: int,
                  out_tokens: Optional[torch.Tensor] = None, n_accepted: Optional[torch.Tensor] = None,
                  workspace: Optional[torch.Tensor] = None, stream=None, pipelined: bool = False):
    """ssd_verify_ragged: per-request gamma [B] int32 and temperature [B] float32.

    pipelined=True calls ssd_verify_ragged_pipelined: the inputs must have been
    complete before the previous verification call on the stream completed."""
    B, W, V = target.shape
    gmax = W - 1
    dev = target.device
    if out_tokens is None:
        out_tokens = torch.empty(B, W, dtype=torch.int32, device=dev)
    if n_accepted is None:
        n_accepted = torch.empty(B, dtype=torch.int32, device=dev)
    ws = _workspace(B, gmax, dev, workspace)
    fn = lib().ssd_verify_ragged_pipelined if pipelined else lib().ssd_verify_ragged
    _check(fn(_dev(target, "target_logits"), _dev(draft, "draft_logits", target.dtype), _dtype_code(target),
              _dev(draft_tokens, "draft_tokens", torch.int32), B, gmax, V, _dev(gamma, "gamma", torch.int32),
              _dev(temperature, "temperature", torch.float32), int(seed) & ((1 << 64) - 1),
              _dev(out_tokens, "out_tokens", torch.int32), _dev(n_accepted, "n_accepted", torch.int32),
              _dev(ws, "workspace"), ws.numel(), _stream(stream)))
    return out_tokens, n_accepted


def saguaro_prespec(target: torch.Tensor, draft: torch.Tensor, k: int, temperature: float, seed: int,
                    bonus_topk: Optional[torch.Tensor] = None, saguaro_tokens: Optional[torch.Tensor] = None,
                    workspace: Optional[torch.Tensor] = None, stream=None, source: str = "residual"):
    """ssd_saguaro_prespec: returns (bonus_topk [B, g+1, k], saguaro_tokens [B, g+1]).
    source: "residual" (top-k of r_j) or "draft" (the draft's k largest logits)."""
    B, W, V = target.shape
    g = W - 1
    dev = target.device
    if bonus_topk is None:
        bonus_topk = torch.empty(B, W, k, dtype=torch.int32, device=dev)
    if saguaro_tokens is None:
        saguaro_tokens = torch.empty(B, W, dtype=torch.int32, device=dev)
    dptr = _dev(draft, "draft_logits", target.dtype) if g > 0 else None
    ws = _saguaro_workspace(B, g, V, dev, workspace)
    _check(lib().ssd_saguaro_prespec(_dev(target, "target_logits"), dptr, _dtype_code(target), B, g, V, int(k),
                                     _source(source), float(temperature), int(seed) & ((1 << 64) - 1),
                                     _dev(bonus_topk, "bonus_topk", torch.int32),
                                     _dev(saguaro_tokens, "saguaro_tokens", torch.int32), _dev(ws, "workspace"),
                                     ws.numel(), _stream(stream)))
    return bonus_topk, saguaro_tokens


def verify_saguaro(target: torch.Tensor, draft: torch.Tensor, draft_tokens: torch.Tensor, k: int,
                   temperature: float, seed: int, workspace: Optional[torch.Tensor] = None, check: bool = True,
                   stream=None, source: str = "residual"):
    """ssd_verify_saguaro: one call for both; returns (out_tokens [B, g+1], n_accepted [B],
    bonus_topk [B, g+1, k], saguaro_tokens [B, g+1], hit [B] or None, n_hits [1] or None)."""
    B, W, V = target.shape
    g = W - 1
    dev = target.device
    out_tokens = torch.empty(B, W, dtype=torch.int32, device=dev)
    n_accepted = torch.empty(B, dtype=torch.int32, device=dev)
    bonus_topk = torch.empty(B, W, k, dtype=torch.int32, device=dev)
    saguaro_tokens = torch.empty(B, W, dtype=torch.int32, device=dev)
    hit = torch.empty(B, dtype=torch.int32, device=dev) if check else None
    n_hits = torch.empty(1, dtype=torch.int32, device=dev) if check else None
    ws = _saguaro_workspace(B, g, V, dev, workspace)
    dptr = _dev(draft, "draft_logits", target.dtype) if g > 0 else None
    tptr = _dev(draft_tokens, "draft_tokens", torch.int32) if g > 0 else None
    _check(lib().ssd_verify_saguaro(_dev(target, "target_logits"), dptr, _dtype_code(target), tptr, B, g, V, int(k),
                                    _source(source), float(temperature), int(seed) & ((1 << 64) - 1), _dev(out_tokens, "out_tokens"),
                                    _dev(n_accepted, "n_accepted"), _dev(bonus_topk, "bonus_topk"),
                                    _dev(saguaro_tokens, "saguaro_tokens"),
                                    _dev(hit, "hit") if check else None, _dev(n_hits, "n_hits") if check else None,
                                    _dev(ws, "workspace"), ws.numel(), _stream(stream)))
    return out_tokens, n_accepted, bonus_topk, saguaro_tokens, hit, n_hits


_topp_ws_cache = {}


def verify_top_p(target: torch.Tensor, draft: Optional[torch.Tensor], draft_tokens: torch.Tensor, temperature: float,
                 top_p: float, seed: int, out_tokens: Optional[torch.Tensor] = None,
                 n_accepted: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None, stream=None):
    """ssd_verify_top_p: both distributions truncated to their top-p nuclei.
    Returns (out_tokens [B, g+1], n_accepted [B])."""
    B, W, V = target.shape
    g = W - 1
    dev = target.device
    if out_tokens is None:
        out_tokens = torch.empty(B, W, dtype=torch.int32, device=dev)
    if n_accepted is None:
        n_accepted = torch.empty(B, dtype=torch.int32, device=dev)
    ws = workspace
    if ws is None:
        key = _ws_key(dev)
        need = int(lib().ssd_verify_top_p_workspace_bytes(B, g))
        ws = _topp_ws_cache.get(key)
        if ws is None or ws.numel() < need:
            ws = torch.zeros(max(need, 1 << 16), dtype=torch.uint8, device=dev)
            _topp_ws_cache[key] = ws
    dptr = _dev(draft, "draft_logits", target.dtype) if draft is not None else None
    tptr = _dev(draft_tokens, "draft_tokens", torch.int32) if g > 0 else None
    _check(lib().ssd_verify_top_p(_dev(target, "target_logits"), dptr, _dtype_code(target), tptr, B, g, V,
                                  float(temperature), float(top_p), int(seed) & ((1 << 64) - 1),
                                  _dev(out_tokens, "out_tokens", torch.int32),
                                  _dev(n_accepted, "n_accepted", torch.int32), _dev(ws, "workspace"), ws.numel(),
                                  _stream(stream)))
    return out_tokens, n_accepted


def verify_saguaro_draft(target: torch.Tensor, draft: torch.Tensor, draft_tokens: torch.Tensor, temperature: float,
                         seed: int, out_tokens: Optional[torch.Tensor] = None,
                         n_accepted: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                         stream=None):
    """ssd_verify_saguaro_draft: draft tokens sampled from each position's Saguaro
    distribution.  Returns (out_tokens [B, g+1], n_accepted [B])."""
    B, W, V = target.shape
    g = W - 1
    dev = target.device
    if out_tokens is None:
        out_tokens = torch.empty(B, W, dtype=torch.int32, device=dev)
    if n_accepted is None:
        n_accepted = torch.empty(B, dtype=torch.int32, device=dev)
    ws = _saguaro_workspace(B, g, V, dev, workspace)
    dptr = _dev(draft, "draft_logits", target.dtype) if g > 0 else None
    tptr = _dev(draft_tokens, "draft_tokens", torch.int32) if g > 0 else None
    _check(lib().ssd_verify_saguaro_draft(_dev(target, "target_logits"), dptr, _dtype_code(target), tptr, B, g, V,
                                          float(temperature), int(seed) & ((1 << 64) - 1),
                                          _dev(out_tokens, "out_tokens", torch.int32),
                                          _dev(n_accepted, "n_accepted", torch.int32), _dev(ws, "workspace"),
                                          ws.numel(), _stream(stream)))
    return out_tokens, n_accepted


def cache_check(bonus_topk: torch.Tensor, out_tokens: torch.Tensor, n_accepted: torch.Tensor, stream=None):
    """ssd_cache_check: (hit [B], n_hits [1])."""
    B, W, k = bonus_topk.shape
    dev = bonus_topk.device
    hit = torch.empty(B, dtype=torch.int32, device=dev)
    n_hits = torch.empty(1, dtype=torch.int32, device=dev)
    _check(lib().ssd_cache_check(_dev(bonus_topk, "bonus_topk", torch.int32), _dev(out_tokens, "out_tokens", torch.int32),
                                 _dev(n_accepted, "n_accepted", torch.int32), B, W - 1, k, _dev(hit, "hit"),
                                 _dev(n_hits, "n_hits"), _stream(stream)))
    return hit, n_hits


def debug_rowstats(target, draft, draft_tokens, temperature, seed, workspace=None, stream=None):
    """ssd_debug_rowstats: (out_tokens, n_accepted, stats [B, g+1, 10] float32)."""
    B, W, V = target.shape
    g = W - 1
    dev = target.device
    out_tokens = torch.empty(B, W, dtype=torch.int32, device=dev)
    n_accepted = torch.empty(B, dtype=torch.int32, device=dev)
    stats = torch.empty(B, W, NSTAT_VERIFY, dtype=torch.float32, device=dev)
    ws = _workspace(B, g, dev, workspace)
    dptr = _dev(draft, "draft_logits", target.dtype) if draft is not None else None
    _check(lib().ssd_debug_rowstats(_dev(target, "target_logits"), dptr, _dtype_code(target),
                                    _dev(draft_tokens, "draft_tokens", torch.int32), B, g, V, float(temperature),
                                    int(seed) & ((1 << 64) - 1), _dev(out_tokens, "out_tokens"),
                                    _dev(n_accepted, "n_accepted"), _dev(stats, "stats"), _dev(ws, "workspace"),
                                    ws.numel(), _stream(stream)))
    return out_tokens, n_accepted, stats


def debug_saguaro_stats(target, draft, k, temperature, seed, workspace=None, stream=None, source="residual"):
    """ssd_debug_saguaro_stats: (bonus_topk, saguaro_tokens, stats [B, g+1, 10])."""
    B, W, V = target.shape
    g = W - 1
    dev = target.device
    bonus_topk = torch.empty(B, W, k, dtype=torch.int32, device=dev)
    saguaro_tokens = torch.empty(B, W, dtype=torch.int32, device=dev)
    stats = torch.empty(B, W, NSTAT_SAGUARO, dtype=torch.float32, device=dev)
    dptr = _dev(draft, "draft_logits", target.dtype) if g > 0 else None
    ws = _saguaro_workspace(B, g, V, dev, workspace)
    _check(lib().ssd_debug_saguaro_stats(_dev(target, "target_logits"), dptr, _dtype_code(target), B, g, V,
                                         int(k), _source(source), float(temperature), int(seed) & ((1 << 64) - 1),
                                         _dev(bonus_topk, "bonus_topk"), _dev(saguaro_tokens, "saguaro_tokens"),
                                         _dev(stats, "stats"), _dev(ws, "workspace"), ws.numel(),
                                         _stream(stream)))
    return bonus_topk, saguaro_tokens, stats


def debug_uniforms(seed: int, B: int, W: int, device=None, stream=None) -> torch.Tensor:
    """ssd_debug_uniforms: [B, W, 3] float32 (accept, resample, Saguaro draws)."""
    out = torch.empty(B, W, 3, dtype=torch.float32, device=device or "cuda")
    _check(lib().ssd_debug_uniforms(int(seed) & ((1 << 64) - 1), B, W, _dev(out, "out"), _stream(stream)))
    return out


def read_status(workspace: Optional[torch.Tensor] = None, device=None, stream=None) -> int:
    """Read and clear the device status word (synchronises the stream)."""
    if workspace is None:
        workspace = _ws_cache.get(_ws_key(device))
        if workspace is None:
            return 0
    st = ctypes.c_int(0)
    _check(lib().ssd_read_status(_dev(workspace, "workspace"), workspace.numel(), ctypes.byref(st),
                                 _stream(stream)))
    return st.value
