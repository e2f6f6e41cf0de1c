"""ssd_verify_noalloc (verification on the library's fixed device scratch)
against ssd_verify with a caller workspace, through the C ABI.

Both entry points run the same kernels with the same Philox draws, so the
tolerance is exact equality of n_accepted and every output token.  Each case
makes two no-alloc calls in a row on one stream before comparing, so the
second call runs on the scratch the first one left behind.  The file is named
to be collected last: it also passes after every other GPU test has run.
"""
import pytest
import torch

from gpu_common import cuda_lib
from speculative_decoding_verification_draft_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

SCRATCH_UNITS = 1600  # B * (gamma + 1) that always fit the 16 MiB scratch


def _outputs(batch):
    B, W = batch.B, batch.gmax + 1
    return (torch.full((B, W), -9, dtype=torch.int32, device="cuda"),
            torch.full((B,), -9, dtype=torch.int32, device="cuda"))


def _two_in_a_row(ssdv, batches, seeds):
    """Two no-alloc calls back to back, then the workspace calls; returns
    [(noalloc outputs, workspace outputs)] per call."""
    outs = [_outputs(b) for b in batches]
    for b, s, (o, n) in zip(batches, seeds, outs):
        ssdv.verify_noalloc(b.target, b.draft, b.draft_tokens, b.temperature, s, o, n)
    torch.cuda.synchronize()
    refs = []
    for b, s in zip(batches, seeds):
        ws = ssdv.make_workspace(b.B, b.gmax)
        refs.append(ssdv.verify(b.target, b.draft, b.draft_tokens, b.temperature, s, workspace=ws))
    torch.cuda.synchronize()
    return list(zip(outs, refs))


def _assert_same(pairs, what):
    for k, ((o, n), (o_ref, n_ref)) in enumerate(pairs):
        assert torch.equal(n, n_ref), f"{what} call {k}: n_accepted differs"
        assert torch.equal(o, o_ref), f"{what} call {k}: out_tokens differ"
        assert (n >= 0).all(), f"{what} call {k}: a request reported an error"


def test_noalloc_matches_workspace_path_bench_shape():
    ssdv = cuda_lib()
    a = wl.zipf_batch(64, 4, 128256, seed=2).to("cuda")
    b = wl.zipf_batch(64, 4, 128256, seed=7).to("cuda")
    _assert_same(_two_in_a_row(ssdv, [a, b], [2, 3]), "B=64 gamma=4 V=128256 bf16")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_noalloc_matches_workspace_path_small_and_greedy(dtype):
    ssdv = cuda_lib()
    sampled = wl.zipf_batch(5, 3, 4099, dtype=dtype, temperature=0.9, seed=11).to("cuda")
    greedy = wl.zipf_batch(6, 2, 1000, dtype=dtype, temperature=0.0, seed=12,
                           sample_tokens=False).to("cuda")
    _assert_same(_two_in_a_row(ssdv, [sampled, greedy], [5, 6]), f"small {dtype}")


def test_noalloc_at_the_scratch_limit():
    ssdv = cuda_lib()
    B, g = 272, 5  # 1632 units: the largest batch at gamma 5
    assert ssdv.workspace_bytes(B, g) <= 16 << 20 < ssdv.workspace_bytes(B + 1, g)
    assert ssdv.workspace_bytes(SCRATCH_UNITS // 32, 31) <= 16 << 20
    a = wl.zipf_batch(B, g, 3001, seed=21).to("cuda")
    b = wl.zipf_batch(B, g, 3001, seed=22).to("cuda")
    _assert_same(_two_in_a_row(ssdv, [a, b], [8, 9]), "B=272 gamma=5")


def test_noalloc_rejects_batches_beyond_the_scratch():
    ssdv = cuda_lib()
    B, g = 64, 31  # 2048 units > 1600
    assert ssdv.workspace_bytes(B, g) > 16 << 20
    batch = wl.zipf_batch(B, g, 64, seed=31).to("cuda")
    o, n = _outputs(batch)
    with pytest.raises(ssdv.SsdError) as err:
        ssdv.verify_noalloc(batch.target, batch.draft, batch.draft_tokens, batch.temperature, 1, o, n)
    assert err.value.status == 9 and str(SCRATCH_UNITS) in str(err.value)
    torch.cuda.synchronize()
    assert (o == -9).all() and (n == -9).all(), "a rejected call must launch nothing"
