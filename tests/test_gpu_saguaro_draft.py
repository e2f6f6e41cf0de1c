"""Verification of draft tokens sampled from the Saguaro distribution
(ssd_verify_saguaro_draft) against the oracle, and its losslessness on the GPU.

p'_i = sqrt(p_i max(r_i, 1e-8)) / sum replaces p_i in the accept test and the
residual (the SSD notes, sections 3.2 and 5.1)."""
import numpy as np
import pytest
import torch

import gpu_common as gc
from speculative_decoding_verification_draft_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ssdv():
    return gc.cuda_lib()


def run(ssdv, batch, T, seed):
    b = batch.to("cuda")
    out, n = ssdv.verify_saguaro_draft(b.target, b.draft, b.draft_tokens, T, seed)
    torch.cuda.synchronize()
    return out.cpu().numpy(), n.cpu().numpy()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("B,gamma,V", [(32, 4, 20000), (16, 1, 4099), (8, 6, 1000), (5, 0, 777), (4, 2, 7)])
def test_matches_oracle(ssdv, dtype, B, gamma, V):
    batch = wl.zipf_batch(B, gamma, V, dtype=dtype, temperature=0.8, seed=V + gamma, sigma_range=(0.3, 1.2))
    out, n = run(ssdv, batch, 0.8, 17)
    ref = gc.verify_oracle(batch, 17, draft_dist="saguaro")
    gc.assert_verify_parity(out, n, ref, V, what=f"saguaro draft B={B} g={gamma} V={V} {dtype}")
    # the mode matters: the plain verification of the same tokens differs somewhere
    if gamma >= 4:
        ref_plain = gc.verify_oracle(batch, 17)
        assert not np.array_equal(ref["n_accepted"], ref_plain["n_accepted"])


def test_saguaro_workload_all_requests(ssdv):
    """B=256, gamma 6, V 152064 fp32 (the Saguaro workload): every request
    against the oracle."""
    batch = wl.zipf_batch(256, 6, 152064, dtype=torch.float32, temperature=0.8, seed=3, sigma_range=(0.6, 0.6))
    out, n = run(ssdv, batch, 0.8, 5)
    ref = gc.verify_oracle(batch, 5, draft_dist="saguaro")
    gc.assert_verify_parity(out, n, ref, 152064, what="saguaro draft, Saguaro workload, all 256 requests")


def test_first_token_follows_target(ssdv):
    """20000 rounds of one request (V 6, gamma 1): x_0 drawn on the host from
    p'_0, verified on the GPU; the first emitted token's histogram matches q_0
    (every bin within 5 sigma), while verifying the same tokens against p does
    not."""
    from scipy.special import softmax
    rng = np.random.default_rng(31)
    V, g, T, B = 6, 1, 0.9, 20000
    xt = rng.normal(0, 1.0, (g + 1, V)).astype(np.float32)
    xd = (xt[:g] + rng.normal(0, 1.5, (g, V))).astype(np.float32)
    q0 = softmax(xt[0].astype(np.float64) / T)
    p0 = softmax(xd[0].astype(np.float64) / T)
    _, psag = gc.orc().saguaro_position(xt[0], xd[0], T)  # the Saguaro distribution of position 0
    tok = rng.choice(V, size=(B, g), p=psag).astype(np.int32)
    target = torch.from_numpy(np.ascontiguousarray(np.broadcast_to(xt, (B, g + 1, V)))).cuda()
    draft = torch.from_numpy(np.ascontiguousarray(np.broadcast_to(xd, (B, g, V)))).cuda()
    toks = torch.from_numpy(tok).cuda()
    out, n = ssdv.verify_saguaro_draft(target, draft, toks, T, 123)
    out_p, _ = ssdv.verify(target, draft, toks, T, 123)
    torch.cuda.synchronize()
    first = out[:, 0].cpu().numpy()
    hist = np.bincount(first, minlength=V) / B
    sd = np.sqrt(q0 * (1 - q0) / B)
    assert np.all(np.abs(hist - q0) < 5 * sd + 1e-12), (hist, q0)
    hist_p = np.bincount(out_p[:, 0].cpu().numpy(), minlength=V) / B
    assert np.any(np.abs(hist_p - q0) > 8 * sd), (hist_p, q0)
