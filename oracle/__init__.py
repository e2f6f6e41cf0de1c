"""fp64 CPU oracle for speculative-decoding verification and Saguaro pre-speculation.

TEST INFRASTRUCTURE ONLY.  The oracle is the plain, slow reference that the CUDA
library is checked against.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.  The
product package never imports it and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C, IEEE fp64, compiled with
``-ffp-contract=off``); this module compiles it with gcc, loads it with ctypes
and marshals numpy arrays.  bf16 logits are passed as their raw ``uint16`` bit
patterns, fp32 logits as ``float32``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "oracle.c")
LIBRARY = os.path.join(HERE, "liboracle.so")

BF16 = 0
F32 = 1
NSTAT_VERIFY = 10
NSTAT_SAGUARO = 10
FLAG_BAND = 1e-6
SAGUARO_CLAMP = 1e-8

_lock = threading.Lock()
_lib = None


def build(out_path: str = LIBRARY, mutant: int = 0) -> str:
    """Compile oracle.c into a shared library (``mutant`` > 0 plants a known bug)."""
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
           f"-DORC_MUTANT={int(mutant)}", "-o", out_path, SOURCE, "-lm", "-pthread"]
    subprocess.run(cmd, check=True)
    return out_path


def _declare(lib):
    c_int, c_double, c_u64, c_float = ctypes.c_int, ctypes.c_double, ctypes.c_uint64, ctypes.c_float
    P = ctypes.c_void_p
    lib.orc_philox4x32_10.argtypes = [P, P, P]
    lib.orc_philox4x32_10.restype = None
    lib.orc_uniform.argtypes = [c_u64, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32]
    lib.orc_uniform.restype = c_double
    lib.orc_uniform_grid.argtypes = [c_u64, c_int, c_int, ctypes.c_uint32, P]
    lib.orc_uniform_grid.restype = None
    lib.orc_softmax.argtypes = [P, c_int, c_double, P, P, P]
    lib.orc_softmax.restype = None
    lib.orc_argmax.argtypes = [P, c_int]
    lib.orc_argmax.restype = c_int
    lib.orc_cache_check.argtypes = [P, P, P, c_int, c_int, c_int, P]
    lib.orc_nucleus.argtypes = [P, P, c_int, c_double, c_double, P]
    lib.orc_nucleus.restype = None
    lib.orc_cache_check.restype = c_int
    lib.orc_choice.argtypes = [P, c_int, c_double, P]
    lib.orc_choice.restype = c_int
    lib.orc_topk.argtypes = [P, c_int, c_int, P, P]
    lib.orc_topk.restype = None
    lib.orc_verify_request.argtypes = [c_int, c_int, P, P, c_double, c_int, c_double, P, P, P, c_double, P, P, P, P]
    lib.orc_verify_request.restype = c_int
    lib.orc_saguaro_request.argtypes = [c_int, c_int, P, P, c_double, c_int, c_int, P, c_double, P, P, P, P, P]
    lib.orc_saguaro_request.restype = c_int
    lib.orc_verify_batch.argtypes = [P, P, c_int, P, c_int, c_int, c_int, P, P, c_float, c_u64,
                                     P, P, P, P, P, P, c_double, c_int, c_int, c_double]
    lib.orc_verify_batch.restype = c_int
    lib.orc_saguaro_batch.argtypes = [P, P, c_int, c_int, c_int, c_int, c_int, c_int, c_float, c_u64,
                                      P, P, P, P, P, P, c_double, c_int]
    lib.orc_saguaro_position.argtypes = [c_int, P, P, c_double, P, P, P, P, P]
    lib.orc_saguaro_position.restype = None
    lib.orc_saguaro_batch.restype = c_int
    lib.orc_draw_row.argtypes = [c_int, c_int, P, P, c_double, c_int, c_double, P, c_int, c_int, c_double,
                                 P, P, P]
    lib.orc_draw_row.restype = c_int
    lib.orc_mutant_id.argtypes = []
    lib.orc_mutant_id.restype = c_int
    return lib


def load(path: Optional[str] = None):
    """Load (building first if needed) the oracle library.  A path loads that build."""
    global _lib
    if path is not None:
        return Oracle(_declare(ctypes.CDLL(path)))
    with _lock:
        if _lib is None:
            stale = (not os.path.exists(LIBRARY)
                     or os.path.getmtime(LIBRARY) < os.path.getmtime(SOURCE))
            if stale:
                build()
            _lib = Oracle(_declare(ctypes.CDLL(LIBRARY)))
    return _lib


def _src(source: str) -> int:
    if source not in ("residual", "draft"):
        raise ValueError(f"top-k source must be 'residual' or 'draft', got {source!r}")
    return 0 if source == "residual" else 1


def _dist(draft_dist: str) -> int:
    if draft_dist not in ("draft", "saguaro"):
        raise ValueError(f"draft distribution must be 'draft' or 'saguaro', got {draft_dist!r}")
    return 0 if draft_dist == "draft" else 1


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _logit_array(a: np.ndarray):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return a, BF16
    if a.dtype == np.float32:
        return a, F32
    raise TypeError(f"logits must be uint16 (bf16 bits) or float32, got {a.dtype}")


class Oracle:
    """numpy-facing wrapper of the C oracle."""

    def __init__(self, lib):
        self.lib = lib
        self.mutant = lib.orc_mutant_id()

    # --- primitives ------------------------------------------------------
    def philox(self, ctr, key) -> np.ndarray:
        ctr = np.ascontiguousarray(ctr, dtype=np.uint32).reshape(-1, 4)
        key = np.ascontiguousarray(key, dtype=np.uint32).reshape(2)
        out = np.empty_like(ctr)
        for n in range(ctr.shape[0]):
            self.lib.orc_philox4x32_10(_ptr(ctr[n]), _ptr(key), _ptr(out[n]))
        return out

    def uniform(self, seed: int, b: int, i: int, d: int) -> float:
        return self.lib.orc_uniform(seed, b, i, d)

    def uniform_grid(self, seed: int, B: int, W: int, d: int) -> np.ndarray:
        out = np.empty((B, W), np.float64)
        self.lib.orc_uniform_grid(seed, B, W, d, _ptr(out))
        return out

    def softmax(self, x, T: float):
        x = np.ascontiguousarray(x, dtype=np.float64)
        prob = np.empty_like(x)
        m, ls = ctypes.c_double(), ctypes.c_double()
        self.lib.orc_softmax(_ptr(x), x.size, T, _ptr(prob), ctypes.byref(m), ctypes.byref(ls))
        return prob, m.value, ls.value

    def argmax(self, x) -> int:
        x = np.ascontiguousarray(x, dtype=np.float64)
        return self.lib.orc_argmax(_ptr(x), x.size)

    def choice(self, w, u: float):
        w = np.ascontiguousarray(w, dtype=np.float64)
        dist = ctypes.c_double()
        k = self.lib.orc_choice(_ptr(w), w.size, u, ctypes.byref(dist))
        return k, dist.value

    def topk(self, w, k: int):
        w = np.ascontiguousarray(w, dtype=np.float64)
        idx = np.empty(k, np.int32)
        val = np.empty(k, np.float64)
        self.lib.orc_topk(_ptr(w), w.size, k, _ptr(idx), _ptr(val))
        return idx, val

    def saguaro_position(self, xt_row, xd_row, T: float, full: bool = False):
        """(r, p_saguaro) of one position; xd_row None at the bonus position.
        full=True also returns q, p_D and the residual mass S."""
        xt = np.ascontiguousarray(xt_row, dtype=np.float64).reshape(-1)
        xd = None if xd_row is None else np.ascontiguousarray(xd_row, dtype=np.float64).reshape(-1)
        r = np.empty_like(xt)
        ps = np.empty_like(xt)
        q = np.empty_like(xt)
        pd = np.empty_like(xt)
        S = ctypes.c_double()
        self.lib.orc_saguaro_position(xt.size, _ptr(xt), _ptr(xd), float(T), _ptr(r), _ptr(ps), _ptr(q),
                                      _ptr(pd), ctypes.byref(S))
        if full:
            return r, ps, q, pd, S.value
        return r, ps

    # --- one request, explicit uniforms ----------------------------------
    def verify_request(self, xt, xd, T, tok, u_acc, u_res, stats: bool = False, band: float = FLAG_BAND,
                       draft_dist: str = "draft", top_p: float = 1.0):
        """xt: (g+1, V) fp64 target logits; xd: (g, V) draft logits; tok: (g,).
        draft_dist: "draft" (tokens sampled from p) or "saguaro" (from the
        Saguaro distribution of each position, which then replaces p)."""
        xt = np.ascontiguousarray(xt, dtype=np.float64)
        g, V = xt.shape[0] - 1, xt.shape[1]
        xd = np.ascontiguousarray(xd, dtype=np.float64).reshape(g, V) if g > 0 else np.zeros((1, V))
        tok = np.ascontiguousarray(tok, dtype=np.int32).reshape(g) if g > 0 else np.zeros(1, np.int32)
        ua = np.ascontiguousarray(u_acc, dtype=np.float64).reshape(-1)
        ur = np.ascontiguousarray(u_res, dtype=np.float64).reshape(-1)
        assert ua.size >= g and ur.size >= g + 1
        out = np.empty(g + 1, np.int32)
        fp, fk = ctypes.c_int32(), ctypes.c_int32()
        st = np.empty((g + 1, NSTAT_VERIFY), np.float64) if stats else None
        n = self.lib.orc_verify_request(g, V, _ptr(xt), _ptr(xd), float(T), _dist(draft_dist), float(top_p),
                                        _ptr(tok), _ptr(ua),
                                        _ptr(ur), float(band), _ptr(out), ctypes.byref(fp),
                                        ctypes.byref(fk), _ptr(st))
        return dict(n=n, out=out, flag_pos=fp.value, flag_kind=fk.value, stats=st)

    def draw_row(self, xt, xd, T, tok, row: int, token: int, band: float = FLAG_BAND, draft_dist: str = "draft",
                 top_p: float = 1.0):
        """(lo, hi, flag_mass) of the draw row `row` of one request (its residual,
        or q_gamma at row == gamma): token's normalised CDF interval [lo, hi) and
        the measure of the uniforms whose draw from this row is flagged."""
        xt = np.ascontiguousarray(xt, dtype=np.float64)
        g, V = xt.shape[0] - 1, xt.shape[1]
        xd = np.ascontiguousarray(xd, dtype=np.float64).reshape(g, V) if g > 0 else np.zeros((1, V))
        tok = np.ascontiguousarray(tok, dtype=np.int32).reshape(g) if g > 0 else np.zeros(1, np.int32)
        lo, hi, fm = ctypes.c_double(), ctypes.c_double(), ctypes.c_double()
        rc = self.lib.orc_draw_row(g, V, _ptr(xt), _ptr(xd), float(T), _dist(draft_dist), float(top_p), _ptr(tok),
                                   int(row), int(token), float(band), ctypes.byref(lo), ctypes.byref(hi),
                                   ctypes.byref(fm))
        if rc != 0:
            raise ValueError("draw_row: greedy request, or row / token out of range")
        return lo.value, hi.value, fm.value

    def saguaro_request(self, xt, xd, T, k, u_sag, stats: bool = False, band: float = FLAG_BAND,
                        source: str = "residual"):
        """source: "residual" (top-k of r_j) or "draft" (top-k of the draft logits,
        the target logits at j = gamma)."""
        xt = np.ascontiguousarray(xt, dtype=np.float64)
        g, V = xt.shape[0] - 1, xt.shape[1]
        xd = np.ascontiguousarray(xd, dtype=np.float64).reshape(g, V) if g > 0 else np.zeros((1, V))
        u = np.ascontiguousarray(u_sag, dtype=np.float64).reshape(-1)
        topk = np.empty((g + 1, k), np.int32)
        tok = np.empty(g + 1, np.int32)
        kf = np.empty(g + 1, np.int32)
        tf = np.empty(g + 1, np.int32)
        st = np.empty((g + 1, NSTAT_SAGUARO), np.float64) if stats else None
        self.lib.orc_saguaro_request(g, V, _ptr(xt), _ptr(xd), float(T), k, _src(source), _ptr(u), float(band),
                                     _ptr(topk), _ptr(tok), _ptr(kf), _ptr(tf), _ptr(st))
        return dict(topk=topk, tokens=tok, topk_flag=kf, tok_flag=tf, stats=st)

    # --- batches over typed logits, Philox uniforms ----------------------
    def verify_batch(self, target, draft, draft_tokens, temperature, seed: int,
                     gamma=None, stats: bool = False, nthreads: int = 1, req_ids=None,
                     band: float = FLAG_BAND, draft_dist: str = "draft", top_p: float = 1.0):
        """target [B, gmax+1, V], draft [B, gmax, V] (uint16 bf16 bits or float32).

        ``temperature``: a float, or a float32 array [B] (per request).
        ``gamma``: None (every request uses gmax) or an int32 array [B].
        ``req_ids``: request index of each row in the Philox counter (default 0..B-1),
        so that a sample of a larger batch draws the same uniforms.
        ``band``: a draw within ``band`` of its threshold or CDF boundary is flagged.
        """
        target, dt = _logit_array(target)
        draft, dd = _logit_array(draft)
        assert dt == dd
        B, W, V = target.shape
        gmax = W - 1
        tok = np.ascontiguousarray(draft_tokens, dtype=np.int32).reshape(B, gmax)
        temps = None
        tscalar = 0.0
        if np.ndim(temperature) == 0:
            tscalar = float(temperature)
        else:
            temps = np.ascontiguousarray(temperature, dtype=np.float32).reshape(B)
        gam = None if gamma is None else np.ascontiguousarray(gamma, dtype=np.int32).reshape(B)
        out = np.empty((B, W), np.int32)
        n = np.empty(B, np.int32)
        fp = np.empty(B, np.int32)
        fk = np.empty(B, np.int32)
        st = np.empty((B, W, NSTAT_VERIFY), np.float64) if stats else None
        rid = None if req_ids is None else np.ascontiguousarray(req_ids, dtype=np.int32).reshape(B)
        rc = self.lib.orc_verify_batch(_ptr(target), _ptr(draft), dt, _ptr(tok), B, gmax, V,
                                       _ptr(gam), _ptr(temps), tscalar, seed, _ptr(out), _ptr(n),
                                       _ptr(fp), _ptr(fk), _ptr(st), _ptr(rid), float(band), nthreads,
                                       _dist(draft_dist), float(top_p))
        if rc != 0:
            raise ValueError("oracle rejected the batch arguments")
        return dict(out_tokens=out, n_accepted=n, flag_pos=fp, flag_kind=fk, stats=st)

    def nucleus(self, x, prob, top_p: float, band: float = FLAG_BAND):
        """(renormalised prob over the top-p nucleus of logits x, ambiguous?)."""
        x = np.ascontiguousarray(x, dtype=np.float64)
        pr = np.array(prob, dtype=np.float64)
        amb = ctypes.c_int(0)
        self.lib.orc_nucleus(_ptr(x), _ptr(pr), x.size, float(top_p), float(band), ctypes.byref(amb))
        return pr, bool(amb.value)

    def cache_check(self, bonus_topk, out_tokens, n_accepted):
        """(hit [B], number of hits) of one round's verify outcome against its
        pre-speculated bonus tokens."""
        topk = np.ascontiguousarray(bonus_topk, dtype=np.int32)
        B, W, k = topk.shape
        out = np.ascontiguousarray(out_tokens, dtype=np.int32).reshape(B, W)
        n = np.ascontiguousarray(n_accepted, dtype=np.int32).reshape(B)
        hit = np.empty(B, np.int32)
        count = self.lib.orc_cache_check(_ptr(topk), _ptr(out), _ptr(n), B, W - 1, k, _ptr(hit))
        return hit, count

    def saguaro_batch(self, target, draft, k: int, temperature: float, seed: int,
                      stats: bool = False, nthreads: int = 1, req_ids=None, band: float = FLAG_BAND,
                      source: str = "residual"):
        target, dt = _logit_array(target)
        draft, dd = _logit_array(draft)
        assert dt == dd
        B, W, V = target.shape
        g = W - 1
        topk = np.empty((B, W, k), np.int32)
        tok = np.empty((B, W), np.int32)
        kf = np.empty((B, W), np.int32)
        tf = np.empty((B, W), np.int32)
        st = np.empty((B, W, NSTAT_SAGUARO), np.float64) if stats else None
        rid = None if req_ids is None else np.ascontiguousarray(req_ids, dtype=np.int32).reshape(B)
        rc = self.lib.orc_saguaro_batch(_ptr(target), _ptr(draft), dt, B, g, V, k, _src(source),
                                        float(temperature), seed, _ptr(topk), _ptr(tok), _ptr(kf),
                                        _ptr(tf), _ptr(st), _ptr(rid), float(band), nthreads)
        if rc != 0:
            raise ValueError("oracle rejected the batch arguments")
        return dict(bonus_topk=topk, saguaro_tokens=tok, topk_flag=kf, tok_flag=tf, stats=st)
