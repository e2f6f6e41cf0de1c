"""The declared limits on the GPU, against the oracle: the largest vocabulary
(SSD_MAX_V = 2^19), the largest gamma (SSD_MAX_GAMMA = 31), the largest top-k
(SSD_MAX_TOPK = 8), both per-lane top-k list lengths of the Saguaro residual
pass (k <= 4 and k > 4), and a batch large enough to be launched as two grid
segments (more than 65535 requests)."""
import numpy as np
import pytest
import torch

import gpu_common as gc
from speculative_decoding_verification_draft_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

MAX_V, MAX_GAMMA, MAX_TOPK = 1 << 19, 31, 8


@pytest.fixture(scope="module")
def ssdv():
    return gc.cuda_lib()


def run_verify(ssdv, batch, seed):
    b = batch.to("cuda")
    out, n = ssdv.verify(b.target, b.draft, b.draft_tokens, b.temperature, seed)
    torch.cuda.synchronize()
    return out.cpu().numpy(), n.cpu().numpy()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_verify_largest_vocabulary(ssdv, dtype):
    """V = 2^19: 32 chunks per row (fp32 rows take the shared-memory form, bf16
    rows the 8-vector register form) and 512 or 1024 pieces per draw row."""
    batch = wl.zipf_batch(3, 2, MAX_V, dtype=dtype, temperature=0.9, seed=91, sigma_range=(0.3, 1.0))
    for seed in (1, 2):
        out, n = run_verify(ssdv, batch, seed)
        gc.assert_verify_parity(out, n, gc.verify_oracle(batch, seed), MAX_V, f"V=2^19 {dtype} seed {seed}")


def test_verify_largest_gamma(ssdv):
    """gamma = 31 draft tokens per request, drafts close to the target so that
    long accepted prefixes occur."""
    batch = wl.zipf_batch(8, MAX_GAMMA, 2000, dtype=torch.bfloat16, temperature=0.8, seed=92, sigma_range=(0.05, 0.3))
    out, n = run_verify(ssdv, batch, 3)
    gc.assert_verify_parity(out, n, gc.verify_oracle(batch, 3), 2000, "gamma 31")
    assert n.max() >= 5


def test_ragged_largest_gamma_with_padding(ssdv):
    """Ragged batch padded to gamma_max = 31: random gammas, some requests
    padded (gamma < 0), half greedy."""
    batch = wl.ragged_batch(24, MAX_GAMMA, 1500, seed=93)
    gam = batch.gamma.clone()
    gam[[2, 9, 17]] = -1
    batch.gamma = gam
    b = batch.to("cuda")
    out, n = ssdv.verify_ragged(b.target, b.draft, b.draft_tokens, b.gamma, b.temperature, 8)
    torch.cuda.synchronize()
    out, n = out.cpu().numpy(), n.cpu().numpy()
    gc.assert_verify_parity(out, n, gc.verify_oracle(batch, 8), 1500, "ragged gamma_max 31")
    assert all(n[r] == -1 and np.all(out[r] == -1) for r in (2, 9, 17))


def test_batch_in_two_grid_segments(ssdv):
    """66000 requests (gamma 0: the bonus draw only), V 300 fp32: the launch is
    split at 65535 requests, and the second segment keeps the requests'
    global indices in the Philox counters."""
    batch = wl.zipf_batch(66000, 0, 300, dtype=torch.float32, temperature=1.0, seed=94)
    out, n = run_verify(ssdv, batch, 5)
    gc.assert_verify_parity(out, n, gc.verify_oracle(batch, 5), 300, "66000 requests")


def saguaro(ssdv, batch, k, T, seed, source="residual"):
    b = batch.to("cuda")
    topk, tok = ssdv.saguaro_prespec(b.target, b.draft, k, T, seed, source=source)
    torch.cuda.synchronize()
    return topk.cpu().numpy(), tok.cpu().numpy()


def test_saguaro_largest_vocabulary_and_k(ssdv):
    """V = 2^19 fp32 with k = 8 (the per-lane top-8 lists), both top-k sources."""
    import test_gpu_saguaro as tgs
    batch = wl.zipf_batch(2, 2, MAX_V, dtype=torch.float32, temperature=0.8, seed=95, sigma_range=(0.6, 0.6),
                          sample_tokens=False)
    for source in ("residual", "draft"):
        topk, tok = saguaro(ssdv, batch, MAX_TOPK, 0.8, 6, source)
        tgs.assert_saguaro_parity(batch, MAX_TOPK, 0.8, 6, topk, tok, what=f"V=2^19 k=8 {source}", source=source)


@pytest.mark.parametrize("k", [4, 5])
def test_saguaro_topk_list_lengths(ssdv, k):
    """k = 4 takes the per-lane top-4 lists of the residual pass, k = 5 the
    top-8 lists: both give the oracle's top-k; and the first four slots of
    k = 5 are the k = 4 result."""
    import test_gpu_saguaro as tgs
    batch = wl.zipf_batch(16, 3, 20000, dtype=torch.float32, temperature=0.8, seed=96, sigma_range=(0.6, 0.6),
                          sample_tokens=False)
    topk, tok = saguaro(ssdv, batch, k, 0.8, 7)
    tgs.assert_saguaro_parity(batch, k, 0.8, 7, topk, tok, what=f"k={k}")
    if k == 5:
        topk4, tok4 = saguaro(ssdv, batch, 4, 0.8, 7)
        assert np.array_equal(topk[:, :, :4], topk4) and np.array_equal(tok, tok4)
