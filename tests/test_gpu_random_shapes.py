"""Random shapes through every entry point, against the oracle.

A fixed, seeded list of configurations: dtype, batch size, gamma up to 31,
vocabularies from 2 to 200000 (bf16 rows of odd length take the
shared-memory form), temperatures including greedy, and one of plain
verification (with the pipelined call, which must give the same outputs),
ragged verification (plain and pipelined), top-p, Saguaro pre-speculation
(either top-k source), the fused call (which must equal the separate calls)
and verification of draft tokens drawn from the Saguaro distribution.  Each case is held to the parity rule of the other GPU tests."""
import random

import pytest
import torch

import gpu_common as gc
from test_gpu_saguaro import assert_saguaro_parity
from speculative_decoding_verification_draft_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

N_CASES = 160
BUDGET = 12_000_000  # elements of one logit tensor per case


def _cases():
    rng = random.Random(20261202)
    out = []
    for _ in range(N_CASES):
        dt = rng.choice([torch.bfloat16, torch.float32])
        V = rng.choice([rng.randint(2, 300), rng.randint(300, 5000), rng.randint(5000, 60000),
                        rng.randint(60000, 200000)])
        if rng.random() < 0.5 and dt == torch.bfloat16 and V % 2 == 0:
            V += 1
        g = rng.choice([0, 1, 2, 3, 4, 5, 6, 8, 12, 16, 31])
        B = rng.randint(1, max(1, min(96, BUDGET // ((g + 1) * V))))
        T = rng.choice([0.0, 0.6, 0.8, 1.0, 1.3])
        kind = rng.choice(["verify", "ragged", "top_p", "saguaro", "fused", "saguaro_draft"])
        extra = dict(top_p=rng.choice([0.3, 0.5, 0.7, 0.9, 0.95, 0.99]), k=rng.randint(1, 8),
                     source=rng.choice(["residual", "draft"]))
        out.append((kind, dt, B, g, V, T, rng.randint(0, 10**9), extra))
    return out


CASES = _cases()


@pytest.fixture(scope="module")
def ssdv():
    return gc.cuda_lib()


@pytest.mark.parametrize("case", range(N_CASES))
def test_random_shape(ssdv, case):
    kind, dt, B, g, V, T, seed, extra = CASES[case]
    what = f"case {case}: {kind} B={B} g={g} V={V} {dt} T={T} seed={seed}"
    data_seed = seed % 1000 + 1
    if kind == "verify":
        b = wl.zipf_batch(B, g, V, dtype=dt, temperature=T, seed=data_seed, sigma_range=(0.3, 1.2),
                          sample_tokens=T > 0)
        db = b.to("cuda")
        o1, n1 = ssdv.verify(db.target, db.draft, db.draft_tokens, T, seed)
        o2, n2 = ssdv.verify_pipelined(db.target, db.draft, db.draft_tokens, T, seed)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(n1, n2), f"{what}: pipelined call differs"
        gc.assert_verify_parity(o1, n1, gc.verify_oracle(b, seed), V, what)
    elif kind == "ragged":
        gm = max(1, g)
        B2 = max(1, min(B, BUDGET // ((gm + 1) * V)))
        b = wl.ragged_batch(B2, gm, V, dtype=dt, seed=data_seed)
        db = b.to("cuda")
        o1, n1 = ssdv.verify_ragged(db.target, db.draft, db.draft_tokens, db.gamma, db.temperature, seed)
        o2, n2 = ssdv.verify_ragged(db.target, db.draft, db.draft_tokens, db.gamma, db.temperature, seed,
                                    pipelined=True)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(n1, n2), f"{what}: pipelined ragged call differs"
        gc.assert_verify_parity(o1, n1, gc.verify_oracle(b, seed), V, what)
    elif kind == "saguaro_draft":
        Ts = T if T > 0 else 0.8
        b = wl.zipf_batch(B, g, V, dtype=dt, temperature=Ts, seed=data_seed, sigma_range=(0.3, 1.2))
        db = b.to("cuda")
        o1, n1 = ssdv.verify_saguaro_draft(db.target, db.draft, db.draft_tokens, Ts, seed)
        torch.cuda.synchronize()
        gc.assert_verify_parity(o1, n1, gc.verify_oracle(b, seed, draft_dist="saguaro"), V, what)
    elif kind == "top_p":
        Tt = T if T > 0 else 0.8
        b = wl.zipf_batch(B, g, V, dtype=dt, temperature=Tt, seed=data_seed, sigma_range=(0.3, 1.2))
        db = b.to("cuda")
        o1, n1 = ssdv.verify_top_p(db.target, db.draft, db.draft_tokens, Tt, extra["top_p"], seed)
        torch.cuda.synchronize()
        gc.assert_verify_parity(o1, n1, gc.verify_oracle(b, seed, top_p=extra["top_p"]), V, what)
    else:  # Saguaro pre-speculation, alone or fused with verification
        g = max(1, g)
        V = max(8, V)
        B = max(1, min(B, BUDGET // ((g + 1) * V)))
        k = min(extra["k"], V)
        Ts = T if T > 0 else 0.8
        b = wl.zipf_batch(B, g, V, dtype=dt, temperature=Ts, seed=data_seed, sigma_range=(0.3, 1.2))
        db = b.to("cuda")
        topk, tok = ssdv.saguaro_prespec(db.target, db.draft, k, Ts, seed, source=extra["source"])
        torch.cuda.synchronize()
        if kind == "fused":
            res = ssdv.verify_saguaro(db.target, db.draft, db.draft_tokens, k, Ts, seed, source=extra["source"])
            o, n = ssdv.verify(db.target, db.draft, db.draft_tokens, Ts, seed)
            torch.cuda.synchronize()
            assert torch.equal(res[0], o) and torch.equal(res[1], n), f"{what}: fused verification differs"
            assert torch.equal(res[2], topk) and torch.equal(res[3], tok), f"{what}: fused Saguaro differs"
        assert_saguaro_parity(b, k, Ts, seed, topk.cpu().numpy(), tok.cpu().numpy(), what=what,
                              source=extra["source"])
