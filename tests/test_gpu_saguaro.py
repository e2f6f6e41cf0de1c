"""GPU Saguaro pre-speculation kernel vs the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import gpu_common as gc
import pins
from speculative_decoding_verification_draft_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOPK_REL, TOPK_ABS = 1e-5, 2e-6


@pytest.fixture(scope="module")
def ssdv():
    return gc.cuda_lib()


def widen(arr, dtype):
    if arr.dtype == np.uint16:
        return (arr.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return arr.astype(np.float64)


# fp32 error scale of a residual entry, relative to (q_v + p_v) / S: a few ulp
# of the exponentials and of the Z_t / Z_d ratio (2^-21 = 8 ulp).
ETA = 2.0 ** -21


def conditioning_bound(r, q, pd, S, bonus):
    """Per-entry bound on |sqrt(p_D max(r, 1e-8))| deviations caused by an
    fp32 residual error delta_v = ETA (q_v + p_D_v) / S.  The square root is
    steep near the 1e-8 clamp, so rows with an entry where q ~ p at large q
    are ill-conditioned; elsewhere the bound is far below 1e-5 Zs."""
    scale = 1.0 if (bonus or S <= 0) else S
    delta = ETA * (q + (0.0 if bonus else pd)) / scale
    s = np.sqrt(pd * np.maximum(r, 1e-8))
    hi = np.sqrt(pd * np.maximum(r + delta, 1e-8))
    lo = np.sqrt(pd * np.maximum(r - delta, 1e-8))
    return np.maximum(hi - s, s - lo)


def assert_saguaro_parity(batch, k, T, seed, topk_g, tok_g, stats_g=None, subset=None, what="", source="residual"):
    """Top-k slots: exact where the oracle does not flag them; where it does,
    the GPU's token must carry (per the oracle) the slot's value within the
    top-k tolerance.  Tokens: exact unless the draw is flagged or lies within
    the row's conditioning bound of a CDF boundary; then the GPU's token must
    own, in the oracle's p_saguaro, an interval that reaches within the band
    plus that bound of the uniform.  The number of flagged draws must match
    the rate the band implies (each draw is flagged with probability
    sum_t min(p_saguaro(t), 2 band)), within 5 binomial sigma.  Statistics:
    log-sums 1e-5, residual mass 1e-5 relative (+2e-6), Zs and p_saguaro of
    the drawn token 1e-5 relative plus the row's conditioning bound."""
    o = gc.orc()
    tgt, dft = batch.numpy_logits()
    idx = np.arange(batch.B) if subset is None else np.asarray(subset)
    ref = o.saguaro_batch(tgt[idx], dft[idx], k, T, seed, stats=stats_g is not None, nthreads=16, req_ids=idx,
                          source=source)
    topk_g = topk_g[idx]
    tok_g = tok_g[idx]
    u = o.uniform_grid(seed, int(idx.max()) + 1, batch.gmax + 1, 2)
    flagged_tok, pred, var = 0, 0.0, 0.0
    g = batch.gmax
    for r_i, b in enumerate(idx):
        for j in range(g + 1):
            bonus = j == g
            rr, ps, q, pd, S = o.saguaro_position(widen(tgt[b, j], tgt.dtype),
                                                  None if bonus else widen(dft[b, j], dft.dtype), T, full=True)
            sv = np.sqrt(pd * np.maximum(rr, 1e-8))
            Zs = sv.sum()
            bound = conditioning_bound(rr, q, pd, S, bonus)
            zs_tol = 1e-5 * Zs + bound.sum()
            want = ref["bonus_topk"][r_i, j]
            got = topk_g[r_i, j]
            flags = ref["topk_flag"][r_i, j]
            for s_ in range(k):
                if flags & (1 << s_):
                    a, c = rr[got[s_]], rr[want[s_]]
                    assert abs(a - c) <= TOPK_REL * c + TOPK_ABS, f"{what}: flagged slot b={b} j={j} s={s_}"
                else:
                    assert got[s_] == want[s_], f"{what}: topk b={b} j={j} slot {s_} gpu {got} oracle {want}"
            t_o, t_g = ref["saguaro_tokens"][r_i, j], tok_g[r_i, j]
            fm = np.minimum(ps, 2 * gc.PAGES_BAND).sum()
            pred += fm
            var += fm * (1 - fm)
            flagged_tok += int(ref["tok_flag"][r_i, j])
            if t_g != t_o:
                cdf = np.cumsum(ps)
                lo, hi = (cdf[t_g - 1] if t_g > 0 else 0.0), cdf[t_g]
                tol = gc.PAGES_BAND + zs_tol / Zs
                assert 0 <= t_g < len(ps) and lo - tol <= u[b, j] < hi + tol, (
                    f"{what}: token b={b} j={j} gpu {t_g} owns [{lo:.9f}, {hi:.9f}) in the oracle's p_saguaro, "
                    f"oracle {t_o}, u {u[b, j]:.9f}, tolerance {tol:.3g}")
            if stats_g is not None:
                sg = stats_g[b, j].astype(np.float64)
                so = ref["stats"][r_i, j]
                assert abs(sg[0] - so[0]) < 1e-5, f"{what}: target log-sum b={b} j={j}"
                if not bonus:
                    assert abs(sg[1] - so[1]) < 1e-5, f"{what}: draft log-sum b={b} j={j}"
                assert abs(sg[2] - so[2]) <= 1e-5 * so[2] + 2e-6, f"{what}: residual mass b={b} j={j}"
                assert abs(sg[3] - so[3]) <= zs_tol, (
                    f"{what}: Zs b={b} j={j} gpu {sg[3]} oracle {so[3]} tol {zs_tol:.3g}")
                if not ref["tok_flag"][r_i, j] and t_g == t_o:
                    rel_tol = 1e-5 + bound[t_o] / sv[t_o] + zs_tol / Zs
                    assert abs(sg[4] / so[4] - 1) <= rel_tol, f"{what}: p_saguaro(token) b={b} j={j}"
                # r_j of the top slot: the fp32 residual e_t - (Z_t/Z_d) e_d cancels where q ~ p, so its
                # error is ETA (q + p) / S (the conditioning model above), not a fraction of r
                scale = 1.0 if (bonus or S <= 0) else S
                r_err = ETA * (q[want[0]] + (0.0 if bonus else pd[want[0]])) / scale
                if source == "draft":
                    r_err = 0.0  # p_j of the top draft logit: no cancellation
                assert abs(sg[5] - so[5]) <= 1e-5 * so[5] + TOPK_ABS + r_err, f"{what}: top-1 value b={b} j={j}"
    # The flag count against the rate the band implies (not the 1e-4 budget:
    # the band covers the whole interval of every token below 2e-6 of mass,
    # a few per cent of the draws for the flat Saguaro mix at V ~ 1.5e5).
    assert abs(flagged_tok - pred) <= 5 * np.sqrt(var) + 2, (
        f"{what}: {flagged_tok} flagged draws, {pred:.1f} expected from the band")


def run(ssdv, batch, k, T, seed, stats=False, source="residual"):
    b = batch.to("cuda")
    if stats:
        topk, tok, st = ssdv.debug_saguaro_stats(b.target, b.draft, k, T, seed, source=source)
        torch.cuda.synchronize()
        return topk.cpu().numpy(), tok.cpu().numpy(), st.cpu().numpy()
    topk, tok = ssdv.saguaro_prespec(b.target, b.draft, k, T, seed, source=source)
    torch.cuda.synchronize()
    return topk.cpu().numpy(), tok.cpu().numpy(), None


def test_toy_tables_topk(ssdv):
    """The page-4 toy tables' residual top-3: token 1 first, then {2, 3}
    (prev 0) / {2, 6} (prev != 0) -- closed forms from the printed tables."""
    t = pins.golden("toy_tables.json")
    lt = np.log(np.array([t["target"]["prev0"], t["target"]["other"]], np.float64)).astype(np.float32)
    ld = np.log(np.array([t["draft"]["prev0"], t["draft"]["other"]], np.float64)).astype(np.float32)
    target = torch.from_numpy(np.stack([np.stack([lt[0], lt[0]]), np.stack([lt[1], lt[1]])]))
    draft = torch.from_numpy(np.stack([ld[0:1], ld[1:2]]))
    batch = wl.Batch(target, draft, torch.zeros(2, 1, dtype=torch.int32), 1.0)
    topk, tok, st = run(ssdv, batch, 3, 1.0, 0, stats=True)
    assert topk[0, 0, 0] == 1 and set(topk[0, 0, 1:]) == {2, 3}
    assert topk[1, 0, 0] == 1 and set(topk[1, 0, 1:]) == {2, 6}
    assert abs(st[0, 0, 2] - 0.05) < 1e-6 and abs(st[1, 0, 2] - 0.04) < 1e-6
    assert abs(st[0, 0, 5] - 0.6) < 1e-5 and abs(st[1, 0, 5] - 0.5) < 1e-5


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("V,gamma,k", [(7, 2, 3), (1000, 3, 1), (4099, 1, 8), (20000, 4, 3), (1, 1, 1)])
def test_small_shapes(ssdv, dtype, V, gamma, k):
    batch = wl.zipf_batch(16, gamma, V, dtype=dtype, temperature=0.8, seed=V, sigma_range=(0.6, 0.6),
                          sample_tokens=False)
    topk, tok, st = run(ssdv, batch, k, 0.8, 21, stats=True)
    assert_saguaro_parity(batch, k, 0.8, 21, topk, tok, st, what=f"V={V} g={gamma} k={k} {dtype}")


def test_equal_distributions(ssdv):
    """q == p at every position: zero residual mass, the residual falls back to q."""
    batch = wl.zipf_batch(8, 3, 3000, seed=5, sample_tokens=False)
    batch.draft.copy_(batch.target[:, :3])
    topk, tok, st = run(ssdv, batch, 3, 0.8, 2, stats=True)
    assert np.all(st[:, :3, 2] == 0)
    assert_saguaro_parity(batch, 3, 0.8, 2, topk, tok, st, what="q == p")


def test_saguaro_config_full_sampled(ssdv):
    """B=256, gamma 6, V 152064 fp32, sigma 0.6, T 0.8, k 3 (the Saguaro workload):
    GPU over the whole batch, oracle on 12 sampled requests."""
    batch = wl.zipf_batch(256, 6, 152064, dtype=torch.float32, temperature=0.8, seed=3, sigma_range=(0.6, 0.6),
                          sample_tokens=False)
    topk, tok, st = run(ssdv, batch, 3, 0.8, 3, stats=True)
    subset = np.random.default_rng(1).choice(256, 12, replace=False)
    assert_saguaro_parity(batch, 3, 0.8, 3, topk, tok, st, subset=subset, what="Saguaro workload")
    # product entry point agrees with the debug entry point
    topk2, tok2, _ = run(ssdv, batch, 3, 0.8, 3)
    assert np.array_equal(topk, topk2) and np.array_equal(tok, tok2)
    # at the pages' vocabulary size every sampled row meets the flat 1e-5 bar
    o = gc.orc()
    tgt, dft = batch.numpy_logits()
    ref = o.saguaro_batch(tgt[subset], dft[subset], 3, 0.8, 3, stats=True, nthreads=16, req_ids=subset)
    rel = np.abs(st[subset, :, 3] / ref["stats"][:, :, 3] - 1)
    assert rel.max() < 1e-5, rel.max()


def test_saguaro_config_full_batch(ssdv):
    """The Saguaro workload (B=256, gamma 6, V 152064 fp32, sigma 0.6, T 0.8,
    k 3) through the product entry point: every request's top-k and Saguaro
    draw against the oracle."""
    batch = wl.zipf_batch(256, 6, 152064, dtype=torch.float32, temperature=0.8, seed=3, sigma_range=(0.6, 0.6),
                          sample_tokens=False)
    topk, tok, _ = run(ssdv, batch, 3, 0.8, 3)
    assert_saguaro_parity(batch, 3, 0.8, 3, topk, tok, what="Saguaro workload, all 256 requests")


def test_segments_and_workspace_reuse(ssdv, monkeypatch):
    """Requests split into segments (each its own streaming, residual and mix
    kernels) give the same outputs as one segment; a workspace reused by a
    smaller shape (whose counters overlap the larger shape's sums) and then by
    the larger shape again changes nothing."""
    batch = wl.zipf_batch(24, 3, 5000, dtype=torch.bfloat16, temperature=0.8, seed=8, sigma_range=(0.6, 0.6),
                          sample_tokens=False)
    small = wl.zipf_batch(2, 1, 300, dtype=torch.float32, temperature=0.8, seed=9, sigma_range=(0.6, 0.6),
                          sample_tokens=False)
    b, s = batch.to("cuda"), small.to("cuda")
    ws = ssdv.make_saguaro_workspace(24, 3, 5000)
    topk_a, tok_a, st_a = ssdv.debug_saguaro_stats(b.target, b.draft, 4, 0.8, 5, workspace=ws)
    topk_a, tok_a, st_a = topk_a.cpu().numpy(), tok_a.cpu().numpy(), st_a.cpu().numpy()
    assert_saguaro_parity(batch, 4, 0.8, 5, topk_a, tok_a, st_a, what="one segment")
    ssdv.saguaro_prespec(s.target, s.draft, 2, 0.8, 1, workspace=ws)
    topk_s, tok_s, st_s = run(ssdv, small, 2, 0.8, 1, stats=True)
    assert_saguaro_parity(small, 2, 0.8, 1, topk_s, tok_s, st_s, what="small shape")
    monkeypatch.setenv("SSDV_SAG_SEGMENT", "5")
    topk_b, tok_b = ssdv.saguaro_prespec(b.target, b.draft, 4, 0.8, 5, workspace=ws)
    torch.cuda.synchronize()
    assert np.array_equal(topk_a, topk_b.cpu().numpy()) and np.array_equal(tok_a, tok_b.cpu().numpy())
    # the same call on a caller stream other than the current one
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        topk_c, tok_c = ssdv.saguaro_prespec(b.target, b.draft, 4, 0.8, 5, workspace=ws, stream=side)
        topk_c, tok_c = topk_c.cpu(), tok_c.cpu()
    assert np.array_equal(topk_a, topk_c.numpy()) and np.array_equal(tok_a, tok_c.numpy())
    assert ssdv.read_status(ws) == 0


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("V,gamma,k", [(7, 2, 3), (4099, 1, 8), (20000, 4, 3), (1, 1, 1)])
def test_draft_source_small_shapes(ssdv, dtype, V, gamma, k):
    """Top-k from the draft logits (the SSD notes' bonus predictor): exact
    against the oracle; the Saguaro draws are those of the residual source."""
    batch = wl.zipf_batch(16, gamma, V, dtype=dtype, temperature=0.8, seed=V + 1, sigma_range=(0.6, 0.6),
                          sample_tokens=False)
    topk, tok, st = run(ssdv, batch, k, 0.8, 21, stats=True, source="draft")
    assert_saguaro_parity(batch, k, 0.8, 21, topk, tok, st, what=f"draft V={V} g={gamma} k={k}", source="draft")
    _, tok_r, _ = run(ssdv, batch, k, 0.8, 21, stats=True)
    assert np.array_equal(tok, tok_r)


def test_draft_source_ties_and_minus_inf(ssdv):
    """Logits rounded to a coarse grid (many equal values: the lower index
    wins) with -inf entries, fewer finite draft logits than k in one row."""
    rng = np.random.default_rng(8)
    B, g, V, k = 4, 2, 300, 8
    xt = np.round(rng.normal(0, 1.0, (B, g + 1, V)), 0).astype(np.float32)
    xd = np.round(rng.normal(0, 1.0, (B, g, V)), 0).astype(np.float32)
    xd[0, 1, :] = -np.inf
    xd[0, 1, [5, 77, 140]] = [0.5, 0.5, -1.0]
    batch = wl.Batch(torch.from_numpy(xt), torch.from_numpy(xd), torch.zeros(B, g, dtype=torch.int32), 1.0)
    topk, tok, st = run(ssdv, batch, k, 1.0, 4, stats=True, source="draft")
    ref = gc.orc().saguaro_batch(xt, xd, k, 1.0, 4, source="draft")
    assert np.array_equal(topk, ref["bonus_topk"]), (topk[0, 1], ref["bonus_topk"][0, 1])
    assert list(topk[0, 1, :3]) == [5, 77, 140]


def test_draft_source_saguaro_workload_sampled(ssdv):
    batch = wl.zipf_batch(256, 6, 152064, dtype=torch.float32, temperature=0.8, seed=3, sigma_range=(0.6, 0.6),
                          sample_tokens=False)
    topk, tok, st = run(ssdv, batch, 3, 0.8, 3, stats=True, source="draft")
    subset = np.random.default_rng(2).choice(256, 8, replace=False)
    assert_saguaro_parity(batch, 3, 0.8, 3, topk, tok, st, subset=subset, what="draft, Saguaro workload",
                          source="draft")
