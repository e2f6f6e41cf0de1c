"""Shared helpers of the GPU parity tests: build/load the CUDA library, run
both implementations on the same bytes, and compare them under the flag rule.

Comparison rule (the oracle's flags): a request with no flagged draw must
match exactly (n_accepted and every output token).  After a flagged draw the
rest of that request is excluded: a flagged resample/bonus draw at position n
still requires the same n and the same accepted prefix; a flagged accept draw
at position f requires only the first f tokens and n >= f.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle

FLAG_RATE_BOUND = 1e-4
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
    return orc().verify_batch(tgt, dft, tok, temps, seed, gamma=gam, stats=stats, nthreads=nthreads,
                              req_ids=req_ids, band=band, draft_dist=draft_dist, top_p=top_p)


def compare_verify(out_g, n_g, ref, V):
    """Returns (mismatched request indices, number of flagged requests, draws)."""
    out_o, n_o, fp, fk = ref["out_tokens"], ref["n_accepted"], ref["flag_pos"], ref["flag_kind"]
    mism, flagged, draws = [], 0, 0
    for b in range(len(n_o)):
        if n_o[b] < 0:
            ok = n_g[b] == -1 and np.all(out_g[b] == -1)
        else:
            draws += int(n_o[b]) + 2
            f = int(fp[b])
            if f < 0:
                ok = n_g[b] == n_o[b] and np.array_equal(out_g[b], out_o[b])
            elif fk[b] == 1:
                flagged += 1
                n = int(n_o[b])
                ok = (n_g[b] == n and np.array_equal(out_g[b][:n], out_o[b][:n])
                      and np.all(out_g[b][n + 1:] == -1) and 0 <= out_g[b][n] < V)
            else:
                flagged += 1
                ok = n_g[b] >= f and np.array_equal(out_g[b][:f], out_o[b][:f])
        if not ok:
            mism.append(b)
    return mism, flagged, draws


def assert_verify_parity(out_g, n_g, ref, V, what="", check_rate=False):
    out_g = out_g.cpu().numpy() if isinstance(out_g, torch.Tensor) else out_g
    n_g = n_g.cpu().numpy() if isinstance(n_g, torch.Tensor) else n_g
    mism, flagged, draws = compare_verify(out_g, n_g, ref, V)
    detail = ""
    if mism:
        b = mism[0]
        detail = (f" first mismatch b={b}: gpu n={n_g[b]} out={out_g[b].tolist()} | oracle "
                  f"n={ref['n_accepted'][b]} out={ref['out_tokens'][b].tolist()} flag="
                  f"({ref['flag_pos'][b]},{ref['flag_kind'][b]})")
    assert not mism, f"{what}: {len(mism)} mismatched requests of {len(n_g)}.{detail}"
    if check_rate:
        assert flagged <= max(1, FLAG_RATE_BOUND * draws), f"{what}: {flagged} flagged of {draws} draws"
    return flagged, draws


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
