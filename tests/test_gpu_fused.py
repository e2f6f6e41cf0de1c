"""Fused verification + Saguaro call and the cache check, through the C ABI.

The fused call must return exactly what the two separate calls return on the
same arguments (both are parity-tested against the oracle on their own), and
its cache check must agree with the oracle's on every request; over many
rounds the hit rate must follow the closed form of the pins."""
import numpy as np
import pytest
import torch

import gpu_common as gc
from speculative_decoding_verification_draft_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ssdv():
    return gc.cuda_lib()


def separate_and_fused(ssdv, b, k, T, seed, source="residual"):
    out_s, n_s = ssdv.verify(b.target, b.draft, b.draft_tokens, T, seed)
    topk_s, tok_s = ssdv.saguaro_prespec(b.target, b.draft, k, T, seed, source=source)
    out_f, n_f, topk_f, tok_f, hit, n_hits = ssdv.verify_saguaro(b.target, b.draft, b.draft_tokens, k, T, seed,
                                                                 source=source)
    torch.cuda.synchronize()
    return [x.cpu().numpy() for x in (out_s, n_s, topk_s, tok_s, out_f, n_f, topk_f, tok_f, hit, n_hits)]


@pytest.mark.parametrize("source", ["residual", "draft"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("B,gamma,V,k", [(24, 4, 20000, 3), (5, 1, 4099, 8), (3, 0, 777, 2), (16, 6, 1000, 1)])
def test_fused_equals_separate_calls(ssdv, dtype, B, gamma, V, k, source):
    batch = wl.zipf_batch(B, gamma, V, dtype=dtype, temperature=0.8, seed=V + B, sigma_range=(0.3, 1.2))
    b = batch.to("cuda")
    out_s, n_s, topk_s, tok_s, out_f, n_f, topk_f, tok_f, hit, n_hits = separate_and_fused(ssdv, b, k, 0.8, 11,
                                                                                           source)
    assert np.array_equal(out_s, out_f) and np.array_equal(n_s, n_f)
    assert np.array_equal(topk_s, topk_f) and np.array_equal(tok_s, tok_f)
    hit_o, count_o = gc.orc().cache_check(topk_f, out_f, n_f)
    assert np.array_equal(hit, hit_o) and int(n_hits[0]) == count_o
    # and the verification itself against the oracle
    gc.assert_verify_parity(out_f, n_f, gc.verify_oracle(batch, 11), V, what=f"fused B={B} g={gamma} V={V}")


def test_fused_saguaro_workload(ssdv):
    """B=256, gamma 6, V 152064 fp32 (the Saguaro workload), draft tokens
    sampled from the draft: fused equals separate over the whole batch."""
    batch = wl.zipf_batch(256, 6, 152064, dtype=torch.float32, temperature=0.8, seed=3, sigma_range=(0.6, 0.6),
                          device="cuda")
    out_s, n_s, topk_s, tok_s, out_f, n_f, topk_f, tok_f, hit, n_hits = separate_and_fused(ssdv, batch, 3, 0.8, 3)
    assert np.array_equal(out_s, out_f) and np.array_equal(n_s, n_f)
    assert np.array_equal(topk_s, topk_f) and np.array_equal(tok_s, tok_f)
    hit_o, count_o = gc.orc().cache_check(topk_f, out_f, n_f)
    assert np.array_equal(hit, hit_o) and int(n_hits[0]) == count_o
    ws = ssdv._sag_ws_cache[ssdv._ws_key("cuda")]
    assert ssdv.read_status(ws) == 0


def test_cache_check_standalone(ssdv):
    """ssd_cache_check on arbitrary outcomes (errors, every n, absent and
    present tokens) equals the oracle's check."""
    rng = np.random.default_rng(5)
    B, g, k, V = 3000, 5, 4, 50
    topk = rng.integers(-1, V, (B, g + 1, k)).astype(np.int32)
    n = rng.integers(-1, g + 1, B).astype(np.int32)
    out = rng.integers(0, V, (B, g + 1)).astype(np.int32)
    for b in range(0, B, 3):  # plant hits
        if n[b] >= 0:
            out[b, n[b]] = topk[b, n[b], rng.integers(0, k)]
    hit, n_hits = ssdv.cache_check(torch.from_numpy(topk).cuda(), torch.from_numpy(out).cuda(),
                                   torch.from_numpy(n).cuda())
    torch.cuda.synchronize()
    hit_o, count_o = gc.orc().cache_check(topk, out, n)
    assert np.array_equal(hit.cpu().numpy(), hit_o) and int(n_hits.item()) == count_o
    assert count_o > B // 4


def test_hit_rate_follows_closed_form(ssdv):
    """20000 rounds of one request (V 6, gamma 2, k 2): the fused call's hit
    rate equals sum_n P(N = n) * (top-k mass of r_n) within 5 sigma."""
    from scipy.special import softmax
    rng = np.random.Generator(np.random.PCG64(21))
    V, g, T, k, B = 6, 2, 0.9, 2, 20000
    xt = rng.normal(0, 1.0, (g + 1, V)).astype(np.float32)
    xd = rng.normal(0, 1.0, (g, V)).astype(np.float32)
    tok = np.array([int(np.argmax(xd[0])), int(np.argsort(xd[1])[-2])], np.int32)
    target = torch.from_numpy(np.ascontiguousarray(np.broadcast_to(xt, (B, g + 1, V)))).cuda()
    draft = torch.from_numpy(np.ascontiguousarray(np.broadcast_to(xd, (B, g, V)))).cuda()
    toks = torch.from_numpy(np.ascontiguousarray(np.broadcast_to(tok, (B, g)))).cuda()
    out, n, topk, stok, hit, n_hits = ssdv.verify_saguaro(target, draft, toks, k, T, 77)
    torch.cuda.synchronize()
    rate = int(n_hits.item()) / B
    q = softmax(xt.astype(np.float64) / T, axis=1)
    p = softmax(xd.astype(np.float64) / T, axis=1)
    a = [min(1.0, q[i, tok[i]] / p[i, tok[i]]) for i in range(g)]
    closed = 0.0
    for j in range(g + 1):
        r = q[g] if j == g else np.maximum(q[j] - p[j], 0.0)
        r = r / r.sum()
        closed += np.prod(a[:j]) * (1.0 - a[j] if j < g else 1.0) * r[np.argsort(-r, kind="stable")[:k]].sum()
    sd = np.sqrt(closed * (1 - closed) / B)
    assert abs(rate - closed) < 5 * sd, (rate, closed, sd)
