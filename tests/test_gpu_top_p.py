"""Verification with top-p (nucleus) truncation on both sides
(ssd_verify_top_p) against the oracle, and its output law on the GPU.

Both the target row q_i and the draft row p_i keep the tokens whose logit is at
least the row's nucleus threshold and are renormalised; the accept test, the
residual and the bonus then run on the truncated distributions (the
verification blog, its closing remark and the section on matching sampling
parameters between target and draft)."""
import numpy as np
import pytest
import torch

import gpu_common as gc
from speculative_decoding_verification_draft_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ssdv():
    return gc.cuda_lib()


def run(ssdv, batch, T, top_p, seed):
    b = batch.to("cuda")
    out, n = ssdv.verify_top_p(b.target, b.draft, b.draft_tokens, T, top_p, seed)
    torch.cuda.synchronize()
    return out.cpu().numpy(), n.cpu().numpy()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("B,gamma,V", [(32, 4, 20000), (16, 1, 4099), (8, 6, 1000), (5, 0, 777), (4, 2, 7)])
@pytest.mark.parametrize("top_p", [0.9, 0.5])
def test_matches_oracle(ssdv, dtype, B, gamma, V, top_p):
    batch = wl.zipf_batch(B, gamma, V, dtype=dtype, temperature=0.8, seed=V + gamma, sigma_range=(0.3, 1.2))
    out, n = run(ssdv, batch, 0.8, top_p, 19)
    ref = gc.verify_oracle(batch, 19, top_p=top_p)
    gc.assert_verify_parity(out, n, ref, V, what=f"top-p {top_p} B={B} g={gamma} V={V} {dtype}")
    # the truncation matters: the plain verification of the same tokens differs somewhere
    if gamma >= 4:
        ref_plain = gc.verify_oracle(batch, 19)
        assert not (np.array_equal(ref["n_accepted"], ref_plain["n_accepted"])
                    and np.array_equal(ref["out_tokens"], ref_plain["out_tokens"]))


def test_emitted_tokens_stay_in_the_target_nucleus(ssdv):
    """Draft tokens drawn from the draft nuclei (as a top-p draft model draws
    them): every emitted token (accepted, correction or bonus) lies in the
    target nucleus of its position, computed on the host from the same
    logits."""
    B, g, V, T, top_p = 64, 4, 5000, 0.8, 0.6
    batch = wl.zipf_batch(B, g, V, dtype=torch.float32, temperature=T, seed=77, sigma_range=(0.3, 1.2))
    o = gc.orc()
    rng = np.random.default_rng(78)

    def nucleus(x):
        x = x.astype(np.float64)
        prob = np.exp((x - x.max()) / T)
        prob /= prob.sum()
        return o.nucleus(x, prob, top_p)[0]

    dft = batch.draft.numpy()
    tok = np.array([[rng.choice(V, p=nucleus(dft[b, i])) for i in range(g)] for b in range(B)], np.int32)
    batch.draft_tokens = torch.from_numpy(tok)
    out, n = run(ssdv, batch, T, top_p, 3)
    tgt = batch.target.numpy()
    for b in range(B):
        for i in range(int(n[b]) + 1):
            assert nucleus(tgt[b, i])[out[b, i]] > 0.0, (b, i, out[b, i])


def test_config3_workload_all_requests(ssdv):
    """B=64, gamma 4, V 128256 bf16 at T 0.8 and top_p 0.9: every request
    against the oracle."""
    batch = wl.zipf_batch(64, 4, 128256, dtype=torch.bfloat16, temperature=0.8, seed=2, sigma_range=(0.3, 1.2))
    out, n = run(ssdv, batch, 0.8, 0.9, 7)
    ref = gc.verify_oracle(batch, 7, top_p=0.9)
    gc.assert_verify_parity(out, n, ref, 128256, what="top-p, B=64 g=4 V=128256, all requests")


def test_open_rows_at_full_size(ssdv):
    """top_p 0.5 at the bench shape leaves about 30 % of the bf16 rows open
    after level 1, so level 2's one-wave kernels walk several (row, chunk)
    items per CTA: every request against the oracle."""
    batch = wl.zipf_batch(64, 4, 128256, dtype=torch.bfloat16, temperature=0.8, seed=3, sigma_range=(0.3, 1.2))
    out, n = run(ssdv, batch, 0.8, 0.5, 11)
    ref = gc.verify_oracle(batch, 11, top_p=0.5)
    gc.assert_verify_parity(out, n, ref, 128256, what="top-p 0.5, B=64 g=4 V=128256, all requests")


def test_top_p_one_and_greedy_are_plain_verification(ssdv):
    """top_p = 1 keeps every token, and greedy rows ignore top_p: both give
    ssd_verify's outputs exactly."""
    batch = wl.zipf_batch(16, 3, 3000, dtype=torch.bfloat16, temperature=0.8, seed=5).to("cuda")
    a = ssdv.verify_top_p(batch.target, batch.draft, batch.draft_tokens, 0.8, 1.0, 11)
    b = ssdv.verify(batch.target, batch.draft, batch.draft_tokens, 0.8, 11)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    a = ssdv.verify_top_p(batch.target, batch.draft, batch.draft_tokens, 0.0, 0.5, 11)
    b = ssdv.verify(batch.target, batch.draft, batch.draft_tokens, 0.0, 11)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_first_token_follows_truncated_target(ssdv):
    """20000 rounds of one request (V 8, gamma 1): x_0 drawn on the host from
    the truncated draft p'_0, verified on the GPU; the first emitted token's
    histogram matches the truncated target q'_0 (every bin within 5 sigma)."""
    rng = np.random.default_rng(41)
    V, g, T, B, top_p = 8, 1, 1.0, 20000, 0.8
    o = gc.orc()
    xt = rng.normal(0, 1.2, (g + 1, V)).astype(np.float32)
    xd = (xt[:g] + rng.normal(0, 1.0, (g, V))).astype(np.float32)

    def truncated(x):
        x = x.astype(np.float64)
        pr = np.exp((x - x.max()) / T)
        pr /= pr.sum()
        kept, amb = o.nucleus(x, pr, top_p)
        assert not amb
        return kept

    q0, p0 = truncated(xt[0]), truncated(xd[0])
    assert (q0 == 0).any() and (p0 == 0).any()  # both truncations bite
    tok = rng.choice(V, size=(B, g), p=p0).astype(np.int32)
    target = torch.from_numpy(np.ascontiguousarray(np.broadcast_to(xt, (B, g + 1, V)))).cuda()
    draft = torch.from_numpy(np.ascontiguousarray(np.broadcast_to(xd, (B, g, V)))).cuda()
    out, _ = ssdv.verify_top_p(target, draft, torch.from_numpy(tok).cuda(), T, top_p, 321)
    torch.cuda.synchronize()
    hist = np.bincount(out[:, 0].cpu().numpy(), minlength=V) / B
    sd = np.sqrt(q0 * (1 - q0) / B)
    assert np.all(np.abs(hist - q0) < 5 * sd + 1e-12), (hist, q0)
