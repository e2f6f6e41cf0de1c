"""Shared helpers of the GPU parity tests: build/load the CUDA library, run
both implementations on the same bytes, and compare them under the flag rule.

Comparison rule.  A request with no flagged draw must match the oracle
exactly (n_accepted and every output token).  A request with a flagged draw
-- a uniform within the band of its accept threshold or of a CDF edge of the
token it drew -- may come out either way at that draw, so it is checked for
validity draw by draw against the oracle's fp64 quantities instead:

  - the first n_gpu output tokens are the draft tokens, the rest after index
    n_gpu are -1;
  - every position the GPU accepted has u_i < a_i + band, and the position
    it rejected has u_i >= a_i - band (a_i the oracle's accept probability);
  - the GPU's correction or bonus token t owns, in the oracle's draw row of
    position n_gpu, an interval [lo, hi) with lo - band <= u' < hi + band
    (every token is valid only when that row's residual mass is below the
    band, where the oracle flags every draw).

So after a flagged draw the rest of the request is still compared: a GPU that
took the other side of a flagged accept draw must draw its correction exactly
as the oracle's fp64 residual of that position allows.  Under top-p, a
position whose nucleus itself is within the band of flipping leaves that
position and the rest of the request unchecked beyond n >= its index.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle

PAGES_BAND = 1e-6  # the pages' band: draws within 1e-6 of a threshold / CDF boundary


def cuda_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_verification_draft_gb300 import build, ssdv
    build.build()
    ssdv.lib()
    return ssdv


def orc():
    return oracle.load()


def widen(arr):
    """Logit rows (bf16 bits as uint16, or float32) as fp64."""
    if arr.dtype == np.uint16:
        return (arr.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return arr.astype(np.float64)


def verify_oracle(batch, seed, stats=False, req_ids=None, subset=None, nthreads=16, band=PAGES_BAND,
                  draft_dist="draft", top_p=1.0):
    tgt, dft = batch.numpy_logits()
    tok = batch.draft_tokens.cpu().numpy()
    temps = batch.temperature
    gam = None if batch.gamma is None else batch.gamma.cpu().numpy()
    if isinstance(temps, torch.Tensor):
        temps = temps.cpu().numpy()
    if subset is not None:
        subset = np.asarray(subset)
        tgt, dft, tok = tgt[subset], dft[subset], tok[subset]
        if gam is not None:
            gam = gam[subset]
        if not np.isscalar(temps) and np.ndim(temps) > 0:
            temps = temps[subset]
        req_ids = subset
    ref = orc().verify_batch(tgt, dft, tok, temps, seed, gamma=gam, stats=stats, nthreads=nthreads,
                             req_ids=req_ids, band=band, draft_dist=draft_dist, top_p=top_p)
    # what the draw-by-draw check of flagged requests needs
    ref["inputs"] = dict(tgt=tgt, dft=dft, tok=tok, temps=temps, gamma=gam, seed=seed,
                         req_ids=np.arange(len(tok)) if req_ids is None else np.asarray(req_ids),
                         band=band, draft_dist=draft_dist, top_p=top_p)
    return ref


def _request(ref, b):
    """One request's fp64 logits, temperature, gamma, tokens and uniforms."""
    inp = ref["inputs"]
    gmax = inp["tok"].shape[1]
    g = gmax if inp["gamma"] is None else int(inp["gamma"][b])
    T = float(inp["temps"]) if np.ndim(inp["temps"]) == 0 else float(inp["temps"][b])
    xt = widen(inp["tgt"][b, :g + 1])
    xd = widen(inp["dft"][b, :g]) if g > 0 else np.zeros((0, xt.shape[1]))
    tok = inp["tok"][b, :g]
    rid = int(inp["req_ids"][b])
    o = orc()
    ua = np.array([o.uniform(inp["seed"], rid, i, 0) for i in range(g + 1)])
    ur = np.array([o.uniform(inp["seed"], rid, i, 1) for i in range(g + 1)])
    return dict(g=g, T=T, xt=xt, xd=xd, tok=tok, ua=ua, ur=ur, band=inp["band"], dist=inp["draft_dist"],
                top_p=inp["top_p"])


def check_flagged(ref, b, out_g, n_g, V):
    """None if the GPU's outcome of flagged request b is valid draw by draw
    (the rule in the module docstring), else the reason."""
    r = _request(ref, b)
    g, band = r["g"], r["band"]
    n = int(n_g)
    W = len(out_g)
    if not 0 <= n <= g:
        return f"n={n} outside [0, {g}]"
    if not np.array_equal(out_g[:n], r["tok"][:n]):
        return "accepted prefix differs from the draft tokens"
    if not np.all(out_g[n + 1:W] == -1):
        return "tokens after the correction are not -1"
    o = orc()
    full = o.verify_request(r["xt"], r["xd"], r["T"], r["tok"], r["ua"], r["ur"], stats=True, band=band,
                            draft_dist=r["dist"], top_p=r["top_p"])
    a = full["stats"][:, 7]
    S = full["stats"][:, 6]
    f, fk = int(ref["flag_pos"][b]), int(ref["flag_kind"][b])
    if r["top_p"] < 1.0 and fk == 0 and abs(r["ua"][f] - a[f]) >= band:
        # the nucleus of position f is itself ambiguous: only what precedes it is fixed
        return None if n >= f else f"n={n} < ambiguous position {f}"
    for i in range(n):
        if not r["ua"][i] < a[i] + band:
            return f"accepted position {i}: u={r['ua'][i]:.9f} >= a={a[i]:.9f} + band"
    if n < g and not r["ua"][n] >= a[n] - band:
        return f"rejected position {n}: u={r['ua'][n]:.9f} < a={a[n]:.9f} - band"
    t = int(out_g[n])
    if not 0 <= t < V:
        return f"token {t} outside [0, {V})"
    if n < g and S[n] < band:
        return None  # a vanishing residual: the oracle flags every draw of this row
    u = r["ur"][n]
    if r["top_p"] < 1.0 and fk == 1 and f == g == n:
        lo_o, hi_o, _ = o.draw_row(r["xt"], r["xd"], r["T"], r["tok"], g, int(ref["out_tokens"][b][g]), band=band,
                                   draft_dist=r["dist"], top_p=r["top_p"])
        if min(u - lo_o, hi_o - u) >= band:
            return None  # the bonus row's nucleus is itself ambiguous: any token of it
    lo, hi, _ = o.draw_row(r["xt"], r["xd"], r["T"], r["tok"], n, t, band=band, draft_dist=r["dist"],
                           top_p=r["top_p"])
    if not (lo - band <= u < hi + band):
        return f"token {t} owns [{lo:.9f}, {hi:.9f}) in row {n}, u'={u:.9f}"
    return None


def request_draws(ref):
    """Draws of each request the oracle verified: one accept uniform per
    position tested (up to the first rejection) and one for the correction or
    bonus; greedy and failed requests draw none."""
    inp = ref["inputs"]
    gmax = inp["tok"].shape[1]
    gam = np.full(len(ref["n_accepted"]), gmax) if inp["gamma"] is None else inp["gamma"]
    temps = np.broadcast_to(np.asarray(inp["temps"], dtype=np.float64), gam.shape)
    n = ref["n_accepted"]
    sampled = (n >= 0) & (temps > 0)
    return np.where(sampled, np.minimum(n + 1, gam) + 1, 0)


def compare_verify(out_g, n_g, ref, V):
    """Returns (mismatched request indices with reasons, number of flagged
    requests, draws)."""
    out_o, n_o, fp = ref["out_tokens"], ref["n_accepted"], ref["flag_pos"]
    mism, flagged = [], 0
    for b in range(len(n_o)):
        why = None
        if n_o[b] < 0:
            if not (n_g[b] == -1 and np.all(out_g[b] == -1)):
                why = "oracle rejects the request, the GPU does not"
        elif int(fp[b]) < 0:
            if not (n_g[b] == n_o[b] and np.array_equal(out_g[b], out_o[b])):
                why = "unflagged request differs"
        else:
            flagged += 1
            why = check_flagged(ref, b, out_g[b], n_g[b], V)
        if why is not None:
            mism.append((b, why))
    return mism, flagged, int(request_draws(ref).sum())


def assert_verify_parity(out_g, n_g, ref, V, what=""):
    out_g = out_g.cpu().numpy() if isinstance(out_g, torch.Tensor) else out_g
    n_g = n_g.cpu().numpy() if isinstance(n_g, torch.Tensor) else n_g
    mism, flagged, draws = compare_verify(out_g, n_g, ref, V)
    detail = ""
    if mism:
        b, why = mism[0]
        detail = (f" first mismatch b={b} ({why}): gpu n={n_g[b]} out={out_g[b].tolist()} | oracle "
                  f"n={ref['n_accepted'][b]} out={ref['out_tokens'][b].tolist()} flag="
                  f"({ref['flag_pos'][b]},{ref['flag_kind'][b]})")
    assert not mism, f"{what}: {len(mism)} mismatched requests of {len(n_g)}.{detail}"
    return flagged, draws


def flag_rate_prediction(ref):
    """(predicted flagged requests, its binomial standard deviation) of the
    oracle's flags on this batch: each sampled request's draw from row n is
    flagged with probability equal to that row's flag mass (the resample
    uniform is independent of the accept draws that fixed n), and each accept
    draw with probability 2 band at most."""
    o = orc()
    pred, var = 0.0, 0.0
    draws = request_draws(ref)
    for b in range(len(ref["n_accepted"])):
        n = int(ref["n_accepted"][b])
        if n < 0 or draws[b] == 0:
            continue
        r = _request(ref, b)
        _, _, fm = o.draw_row(r["xt"], r["xd"], r["T"], r["tok"], n, int(ref["out_tokens"][b][n]),
                              band=r["band"], draft_dist=r["dist"], top_p=r["top_p"])
        pa = min(1.0, 2 * r["band"] * (draws[b] - 1))
        p = fm + pa - fm * pa
        pred += p
        var += p * (1 - p)
    return pred, float(np.sqrt(var))


def edge_errors(st_g, ref, out_g):
    """|GPU - oracle| of the normalised CDF edges of every token both sides drew
    identically (same n, same token), measured as the uniform's distance to
    each edge."""
    st_g = st_g.cpu().numpy().astype(np.float64) if isinstance(st_g, torch.Tensor) else st_g
    out_g = out_g.cpu().numpy() if isinstance(out_g, torch.Tensor) else out_g
    so = ref["stats"]
    errs = []
    for b in range(len(ref["n_accepted"])):
        n = int(ref["n_accepted"][b])
        if n < 0 or out_g[b][n] != ref["out_tokens"][b][n]:
            continue
        for c in (8, 9):
            if np.isfinite(so[b, n, c]) and np.isfinite(st_g[b, n, c]):
                errs.append(abs(st_g[b, n, c] - so[b, n, c]))
    return np.array(errs)


def assert_stats_close(st_g, st_o, greedy=False, what=""):
    """Per-position statistics: softmax log-sums within 1e-5, token
    probabilities within 1e-5 relative, residual mass within 1e-5 relative
    plus an absolute floor of 2e-6 (fp32 cancellation in q - p), accept
    probability within 1e-6."""
    st_g = st_g.cpu().numpy().astype(np.float64)
    g = st_g.shape[1] - 1
    if greedy:
        assert np.array_equal(st_g[:, :, 0], st_o[:, :, 0]), f"{what}: row max"
        return
    assert np.array_equal(st_g[:, :, 0], st_o[:, :, 0]), f"{what}: target row max"
    assert np.abs(st_g[:, :, 1] - st_o[:, :, 1]).max() < 1e-5, f"{what}: target log-sum"
    if g == 0:
        return
    s_g, s_o = st_g[:, :g], st_o[:, :g]
    assert np.array_equal(s_g[:, :, 2], s_o[:, :, 2]), f"{what}: draft row max"
    assert np.abs(s_g[:, :, 3] - s_o[:, :, 3]).max() < 1e-5, f"{what}: draft log-sum"
    for col, name in [(4, "q(x)"), (5, "p(x)")]:
        rel = np.abs(s_g[:, :, col] - s_o[:, :, col]) / np.maximum(s_o[:, :, col], 1e-30)
        ok = (rel < 1e-5) | (np.abs(s_g[:, :, col] - s_o[:, :, col]) < 1e-12)
        assert ok.all(), f"{what}: {name} max rel {rel.max()}"
    dS = np.abs(s_g[:, :, 6] - s_o[:, :, 6])  # residual mass
    assert (dS <= 1e-5 * s_o[:, :, 6] + 2e-6).all(), f"{what}: residual mass max diff {dS.max()}"
    assert np.abs(s_g[:, :, 7] - s_o[:, :, 7]).max() < 1e-6, f"{what}: accept probability"
