"""Pins of the CPU oracle to facts fixed by the pages and by mathematics.

Each ``pin_*`` function takes an oracle instance and raises AssertionError when
the oracle disagrees with a value the pages print, a closed form, an invariant
or an independent library routine.  ``test_oracle_pins.py`` runs them on the
real oracle; ``test_oracle_mutants.py`` builds the oracle with a planted
mistake and checks that at least one pin fails.

Nothing here recomputes the oracle's own formula: expected values come from
the pages' tables (``golden/``), from closed forms (losslessness: the emitted
law equals the target; acceptance probability = sum min(p, q); E[N]), or from
library routines (scipy softmax / logsumexp, numpy argmax / argsort /
searchsorted, triton's Philox4x32-10).
"""
from __future__ import annotations

import functools
import json
import os
import subprocess
import sys
from collections import defaultdict

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def toy_tables():
    t = golden("toy_tables.json")
    return (np.array(t["draft"]["prev0"]), np.array(t["draft"]["other"]),
            np.array(t["target"]["prev0"]), np.array(t["target"]["other"]))


# --------------------------------------------------------------------------
# Philox4x32-10 against triton's implementation (run in its CPU interpreter)
# --------------------------------------------------------------------------

_TRITON_SCRIPT = r"""
import os, sys, json
os.environ["TRITON_INTERPRET"] = "1"
import torch, triton, triton.language as tl

@triton.jit
def kern(out_ptr, c0p, c1p, c2p, c3p, seed, N: tl.constexpr):
    o = tl.arange(0, N)
    a, b, c, d = tl.philox(seed, tl.load(c0p + o), tl.load(c1p + o), tl.load(c2p + o), tl.load(c3p + o))
    tl.store(out_ptr + o * 4 + 0, a)
    tl.store(out_ptr + o * 4 + 1, b)
    tl.store(out_ptr + o * 4 + 2, c)
    tl.store(out_ptr + o * 4 + 3, d)

req = json.loads(sys.stdin.read())
res = []
for item in req:
    ctr = torch.tensor(item["ctr"], dtype=torch.int64).to(torch.int32).reshape(-1, 4)
    n = ctr.shape[0]
    cols = [ctr[:, j].contiguous() for j in range(4)]
    out = torch.zeros(n * 4, dtype=torch.int32)
    kern[(1,)](out, *cols, item["seed"], n)
    res.append([(x & 0xffffffff) for x in out.tolist()])
print(json.dumps(res))
"""


def philox_cases():
    rng = np.random.Generator(np.random.PCG64(1234))
    cases = []
    seeds = [0, 1, 0xFFFFFFFF, 0x123456789ABCDEF0, (1 << 64) - 1, 42]
    for s in seeds:
        ctr = rng.integers(0, 1 << 32, size=(32, 4), dtype=np.uint64)
        ctr[0] = 0
        ctr[1] = [0xFFFFFFFF] * 4
        ctr[2] = [0, 1, 0, 0]
        cases.append((s, ctr.astype(np.uint32)))
    return cases


@functools.lru_cache(maxsize=1)
def triton_philox_reference():
    """Outputs of triton.language.philox (key = seed lo/hi, 10 rounds)."""
    req = []
    for s, ctr in philox_cases():
        # triton takes the seed as a signed 64-bit scalar; pass its two's complement
        sv = s if s < (1 << 63) else s - (1 << 64)
        req.append({"seed": sv, "ctr": [int(x) for x in ctr.reshape(-1)]})
    env = dict(os.environ, TRITON_INTERPRET="1")
    p = subprocess.run([sys.executable, "-c", _TRITON_SCRIPT], input=json.dumps(req),
                       capture_output=True, text=True, env=env, timeout=600)
    if p.returncode != 0:
        raise RuntimeError("triton interpreter failed: " + p.stderr[-2000:])
    return [np.array(r, dtype=np.uint64).reshape(-1, 4) for r in json.loads(p.stdout)]


def pin_philox_vs_triton(o):
    ref = triton_philox_reference()
    for (s, ctr), want in zip(philox_cases(), ref):
        key = np.array([s & 0xFFFFFFFF, s >> 32], np.uint64).astype(np.uint32)
        got = o.philox(ctr, key).astype(np.uint64)
        assert np.array_equal(got, want), f"Philox mismatch for seed {s:#x}"


def pin_uniform_mapping(o):
    """u = (word >> 8) * 2^-24 of word (d mod 4) of Philox(counter (b, i, d/4, 0))."""
    for (seed, b, i, d) in [(0, 0, 0, 0), (7, 3, 2, 1), (2**40 + 5, 100, 8, 2), (1, 5, 5, 5)]:
        key = np.array([seed & 0xFFFFFFFF, seed >> 32], np.uint64).astype(np.uint32)
        w = o.philox(np.array([[b, i, d >> 2, 0]], np.uint32), key)[0, d & 3]
        assert o.uniform(seed, b, i, d) == float(int(w) >> 8) * 2.0**-24


def pin_uniform_statistics(o, n_b=4096, n_i=64):
    u = o.uniform_grid(99, n_b, n_i, 1).reshape(-1)
    n = u.size
    assert np.all(u >= 0) and np.all(u < 1)
    assert np.all(u * 2**24 == np.floor(u * 2**24))
    assert abs(u.mean() - 0.5) < 5 * np.sqrt(1 / 12 / n)
    hist = np.bincount(np.minimum((u * 256).astype(int), 255), minlength=256)
    chi2 = ((hist - n / 256) ** 2 / (n / 256)).sum()
    assert chi2 < 255 + 6 * np.sqrt(2 * 255), chi2
    c = np.corrcoef(u[:-1], u[1:])[0, 1]
    assert abs(c) < 5 / np.sqrt(n), c


# --------------------------------------------------------------------------
# Softmax, argmax, top-k, inverse CDF against library routines / invariants
# --------------------------------------------------------------------------

def pin_softmax(o):
    from scipy.special import logsumexp, softmax
    rng = np.random.Generator(np.random.PCG64(5))
    for V, T in [(7, 1.0), (100, 0.8), (1000, 0.3), (33, 2.5)]:
        x = rng.normal(0, 3, V)
        p, m, ls = o.softmax(x, T)
        assert m == x.max()
        assert np.allclose(p, softmax(x / T), rtol=1e-12, atol=0)
        assert abs(ls - logsumexp((x - x.max()) / T)) < 1e-12
        # shift invariance and closed-form ratios
        p2, _, _ = o.softmax(x + 17.25, T)
        assert np.allclose(p, p2, rtol=1e-12, atol=0)
        a, b = 0, V - 1
        assert abs(p[a] / p[b] - np.exp((x[a] - x[b]) / T)) < 1e-12 * np.exp((x[a] - x[b]) / T)


def pin_argmax(o):
    rng = np.random.Generator(np.random.PCG64(6))
    for V in [1, 2, 7, 1000]:
        for _ in range(20):
            x = rng.integers(-3, 4, V).astype(np.float64)  # many ties
            assert o.argmax(x) == int(np.argmax(x))


def pin_topk(o):
    rng = np.random.Generator(np.random.PCG64(7))
    for V, k in [(7, 3), (50, 5), (200, 8), (5, 5)]:
        for _ in range(10):
            w = rng.integers(0, 6, V).astype(np.float64) / 5.0  # ties
            idx, val = o.topk(w, k)
            want = np.argsort(-w, kind="stable")[:k]
            assert np.array_equal(idx, want), (idx, want)
            assert np.array_equal(val, w[want])


def pin_choice(o):
    rng = np.random.Generator(np.random.PCG64(8))
    for V in [1, 7, 64]:
        for _ in range(10):
            w = rng.random(V) * (rng.random(V) < 0.6)
            if w.sum() == 0:
                w[V // 2] = 1.0
            c = np.cumsum(w)
            S = c[-1]
            for u in np.concatenate([rng.random(50), [0.0, 1 - 2**-24]]):
                k, _ = o.choice(w, u)
                want = int(np.searchsorted(c, u * S, side="right"))
                if want >= V:  # rounding fallback: last positive entry
                    want = int(np.nonzero(w)[0][-1])
                assert k == want, (k, want)
            # every positive-weight token owns the interval [C_{k-1}/S, C_k/S)
            for k in np.nonzero(w)[0]:
                lo = (c[k - 1] if k > 0 else 0.0) / S
                hi = c[k] / S
                got, dist = o.choice(w, 0.5 * (lo + hi))
                assert got == k
                assert abs(dist - 0.5 * (hi - lo)) < 1e-12


# --------------------------------------------------------------------------
# Exact laws by enumeration of the oracle's decision function
# --------------------------------------------------------------------------

def step_law(f, lo=0.0, hi=1.0, tol=2.0**-44):
    """Pieces (value, a, b) of a monotone step function f on [lo, hi)."""
    pieces = []

    def rec(a, fa, b, fb):
        if fa == fb:
            pieces.append((fa, a, b))
            return
        if b - a < tol:
            m = 0.5 * (a + b)
            pieces.append((fa, a, m))
            pieces.append((fb, m, b))
            return
        m = 0.5 * (a + b)
        fm = f(m)
        rec(a, fa, m, fm)
        rec(m, fm, b, fb)

    top = np.nextafter(hi, lo)
    rec(lo, f(lo), top, f(top))
    # merge adjacent equal pieces
    out = []
    for v, a, b in pieces:
        if out and out[-1][0] == v:
            out[-1] = (v, out[-1][1], b)
        else:
            out.append((v, a, b))
    return out


def request_law(o, xt, xd, T, tok, **kw):
    """{emitted tuple: probability} of one request, over its uniforms."""
    g = len(tok)
    law = defaultdict(float)

    def run(ua, ur):
        return o.verify_request(xt, xd, T, tok, ua, ur, **kw)

    def explore(i, ua, weight):
        ur = np.full(g + 1, 0.5)
        if i == g:
            for val, a, b in step_law(lambda u: tuple(run(ua, np.where(np.arange(g + 1) == g, u, ur))["out"])):
                law[val] += weight * (b - a)
            return
        def accepted(u):
            ua2 = ua.copy()
            ua2[i] = u
            return run(ua2, ur)["n"] > i
        for acc, a, b in step_law(accepted):
            ua2 = ua.copy()
            ua2[i] = 0.5 * (a + b)
            if acc:
                explore(i + 1, ua2, weight * (b - a))
            else:
                for val, c, d in step_law(lambda u: tuple(run(ua2, np.where(np.arange(g + 1) == i, u, ur))["out"])):
                    law[val] += weight * (b - a) * (d - c)

    explore(0, np.full(max(g, 1), 0.5), 1.0)
    return law


def emitted(out):
    return tuple(int(t) for t in out if t >= 0)


def pin_toy_closed_forms(o):
    """The blog's toy tables: alpha = sum min(p, q) = 0.95 (prev 0) / 0.96 (else);
    residual (q-p)+/S = [0,.6,.2,.2,0,0,0] / [0,.5,.25,0,0,0,.25]."""
    d0, d1, t0, t1 = toy_tables()
    for p, q, alpha, resid in [(d0, t0, 0.95, [0, .6, .2, .2, 0, 0, 0]),
                               (d1, t1, 0.96, [0, .5, .25, 0, 0, 0, .25])]:
        xt = np.log(np.stack([q, q]))
        xd = np.log(p)[None]
        # P(accept at position 0) = sum_x p(x) * P(u < a(x))
        pa = 0.0
        resid_law = np.zeros(7)
        for x in range(7):
            law = request_law(o, xt, xd, 1.0, [x])
            acc = sum(v for k, v in law.items() if len(emitted(k)) == 2)
            pa += p[x] * acc
            for k, v in law.items():
                e = emitted(k)
                if len(e) == 1:
                    resid_law[e[0]] += p[x] * v
        assert abs(pa - alpha) < 1e-9, (pa, alpha)
        assert np.allclose(resid_law / resid_law.sum(), resid, atol=1e-9), resid_law
        st = o.verify_request(xt, xd, 1.0, [1], [0.5], [0.5, 0.5], stats=True)["stats"]
        assert abs(st[0, 6] - (1 - alpha)) < 1e-9


def pin_losslessness_toy_chain(o, gamma=2):
    """Exact law of one round on the toy Markov model equals the target chain:
    the first emitted token ~ q(.|0), and each next token, given the emitted
    prefix and that the round reached it, ~ q(.|previous token)."""
    d0, d1, t0, t1 = toy_tables()
    V = 7
    dist = lambda prev, tab0, tab1: tab0 if prev == 0 else tab1
    joint = defaultdict(float)
    import itertools
    for xs in itertools.product(range(V), repeat=gamma):
        w = 1.0
        prev = 0
        for x in xs:
            w *= dist(prev, d0, d1)[x]
            prev = x
        prevs = [0] + list(xs)
        xt = np.log(np.stack([dist(pv, t0, t1) for pv in prevs]))
        xd = np.log(np.stack([dist(pv, d0, d1) for pv in prevs[:gamma]]))
        for k, v in request_law(o, xt, xd, 1.0, list(xs)).items():
            joint[emitted(k)] += w * v
    assert abs(sum(joint.values()) - 1) < 1e-9
    # prefix masses: P(y_0..y_{m-1}, round emits >= m tokens)
    prefix = defaultdict(float)
    for seq, pr in joint.items():
        for m in range(1, len(seq) + 1):
            prefix[seq[:m]] += pr
    first = np.array([prefix[(v,)] for v in range(V)])
    assert np.allclose(first, t0, atol=1e-9), first
    for pre, pm in list(prefix.items()):
        if len(pre) >= gamma + 1 or pm < 1e-12:
            continue
        nxt = np.array([prefix.get(pre + (w,), 0.0) for w in range(V)])
        if nxt.sum() == 0:
            continue
        cond = nxt / nxt.sum()
        want = dist(pre[-1], t0, t1)
        assert np.allclose(cond, want, atol=1e-8), (pre, cond, want)
    # P(first draft accepted) = sum min(p, q) at prev 0
    p_reach2 = sum(pr for seq, pr in joint.items() if len(seq) >= 2)
    assert abs(p_reach2 - 0.95) < 1e-9


def pin_losslessness_random(o):
    """Position-dependent random distributions (not Markov), gamma = 2, T != 1:
    y_0 ~ q_0; given reached, y_1 ~ q_1 and the bonus y_2 ~ q_2."""
    from scipy.special import softmax
    rng = np.random.Generator(np.random.PCG64(11))
    V, g, T = 5, 2, 0.7
    xt = rng.normal(0, 1.5, (g + 1, V))
    xd = xt[:g] + rng.normal(0, 0.8, (g, V))
    q = softmax(xt / T, axis=1)
    p = softmax(xd / T, axis=1)
    import itertools
    joint = defaultdict(float)
    for xs in itertools.product(range(V), repeat=g):
        w = p[0, xs[0]] * p[1, xs[1]]
        for k, v in request_law(o, xt, xd, T, list(xs)).items():
            joint[emitted(k)] += w * v
    prefix = defaultdict(float)
    for seq, pr in joint.items():
        for m in range(1, len(seq) + 1):
            prefix[seq[:m]] += pr
    assert np.allclose([prefix[(v,)] for v in range(V)], q[0], atol=1e-9)
    for pre, pm in list(prefix.items()):
        if len(pre) > g or pm < 1e-12:
            continue
        nxt = np.array([prefix.get(pre + (w,), 0.0) for w in range(V)])
        if nxt.sum() == 0:
            continue
        assert np.allclose(nxt / nxt.sum(), q[len(pre)], atol=1e-8)
    acc0 = sum(pr for seq, pr in joint.items() if len(seq) >= 2)
    assert abs(acc0 - np.minimum(p[0], q[0]).sum()) < 1e-9


def pin_greedy(o):
    """Greedy (T = 0) reduces to argmax matching (numpy argmax, first index)."""
    rng = np.random.Generator(np.random.PCG64(12))
    for _ in range(40):
        g, V = int(rng.integers(1, 5)), int(rng.integers(1, 9))
        xt = rng.integers(-2, 3, (g + 1, V)).astype(np.float64)
        am = xt.argmax(axis=1)
        tok = np.where(rng.random(g) < 0.7, am[:g], rng.integers(0, V, g))
        r = o.verify_request(xt, np.zeros((g, V)), 0.0, tok, np.zeros(g), np.zeros(g + 1))
        mism = np.nonzero(tok != am[:g])[0]
        n = int(mism[0]) if mism.size else g
        assert r["n"] == n
        want = list(tok[:n]) + [am[n]]
        assert list(r["out"][:n + 1]) == want and all(r["out"][n + 1:] == -1)


def pin_low_temperature_limit(o):
    """As T -> 0+, sampled verification agrees with greedy on separated logits:
    position 0 proposes the target argmax (accepted), position 1 proposes a
    token the draft is sure of but the target is not (rejected, corrected to
    the target argmax)."""
    rng = np.random.Generator(np.random.PCG64(13))
    for _ in range(20):
        g, V = 3, 6
        xt = rng.permuted(np.tile(np.arange(V, dtype=np.float64), (g + 1, 1)), axis=1)
        xd = xt[:g].copy()
        tok = xt[:g].argmax(axis=1)
        tok[1] = (tok[1] + 1) % V
        xd[1, tok[1]] = xt[1].max() + 1.0
        u = rng.random(g + 1) * 0.98 + 0.01
        s = o.verify_request(xt, xd, 1e-3, tok, u[:g], u)
        gr = o.verify_request(xt, xd, 0.0, tok, u[:g], u)
        assert s["n"] == gr["n"] == 1
        assert list(s["out"]) == list(gr["out"])
        assert s["out"][1] == xt[1].argmax()


def pin_expected_tokens(o):
    """E[N] = (1 - a^(g+1)) / (1 - a) tokens per round for i.i.d. positions,
    a = sum min(p, q) (blog §4), by Monte-Carlo within 4 standard errors."""
    from scipy.special import softmax
    rng = np.random.Generator(np.random.PCG64(14))
    V, g, B, T = 16, 4, 60000, 0.7
    zt = rng.normal(0, 1.2, V)
    zd = zt + rng.normal(0, 0.6, V)
    q, p = softmax(zt / T), softmax(zd / T)
    alpha = np.minimum(p, q).sum()
    target = np.broadcast_to(zt.astype(np.float32), (B, g + 1, V)).copy()
    draft = np.broadcast_to(zd.astype(np.float32), (B, g, V)).copy()
    p32 = softmax(draft[0, 0].astype(np.float64) / T)
    tok = rng.choice(V, size=(B, g), p=p32 / p32.sum()).astype(np.int32)
    r = o.verify_batch(target, draft, tok, T, seed=3, nthreads=4)
    N = r["n_accepted"] + 1
    EN = (1 - alpha ** (g + 1)) / (1 - alpha)
    se = N.std() / np.sqrt(B)
    assert abs(N.mean() - EN) < 4 * se, (N.mean(), EN, se)


def toy_verify_batch(o, B, gamma=4, seed=0, tok_seed=0):
    d0, d1, t0, t1 = toy_tables()
    tables = {"draft": {"prev0": list(d0), "other": list(d1)},
              "target": {"prev0": list(t0), "other": list(t1)}}
    from speculative_decoding_verification_draft_gb300 import workloads
    bt = workloads.toy_batch(tables, B, gamma, tok_seed)
    tgt, dft = bt.numpy_logits()
    r = o.verify_batch(tgt, dft, bt.draft_tokens.numpy(), 1.0, seed=seed, nthreads=8)
    return r


def kl(pemp, q):
    m = pemp > 0
    return float((pemp[m] * np.log(pemp[m] / q[m])).sum())


def pin_toy_kl(o, draws=200000):
    """The blog's unbiasedness check: 200k speculative draws on the toy model,
    histogram vs the target; the page reports KL ~ 4.5e-5 (bound 1e-4)."""
    info = golden("unbiasedness_check.json")
    _, _, t0, t1 = toy_tables()
    r = toy_verify_batch(o, draws)
    out, n = r["out_tokens"], r["n_accepted"]
    first = np.bincount(out[:, 0], minlength=7) / draws
    assert kl(first, t0) < info["kl_bound"], kl(first, t0)
    assert np.abs(first - t0).max() < 0.005
    # transitions inside rounds: prev -> next among emitted tokens
    pairs0, pairs1 = np.zeros(7), np.zeros(7)
    for k in range(1, out.shape[1]):
        ok = n >= k
        prev, nxt = out[ok, k - 1], out[ok, k]
        pairs0 += np.bincount(nxt[prev == 0], minlength=7)
        pairs1 += np.bincount(nxt[prev != 0], minlength=7)
    assert kl(pairs0 / pairs0.sum(), t0) < info["kl_bound"]
    assert kl(pairs1 / pairs1.sum(), t1) < info["kl_bound"]


def pin_speedup_formula():
    """The blog's §4 table equals E[N]/(gamma c + 1) to 2 d.p., except the
    misprinted alpha=0.5, gamma=5 cell."""
    t = golden("speedup_table.json")
    bad = {(m["alpha"], m["c"], m["gamma"]) for m in t["misprinted"]}
    for row in t["rows"]:
        a, c = row["alpha"], row["c"]
        for gm, printed in zip(t["gammas"], row["speedup"]):
            s = (1 - a ** (gm + 1)) / (1 - a) / (gm * c + 1)
            if (a, c, gm) in bad:
                assert abs(s - printed) > 0.05
            else:
                assert abs(s - printed) <= 0.0051, (a, c, gm, s, printed)


# --------------------------------------------------------------------------
# Saguaro pins
# --------------------------------------------------------------------------

def sag_token_law(o, xt, xd, T, j):
    g = xt.shape[0] - 1

    def f(u):
        us = np.full(g + 1, 0.5)
        us[j] = u
        return int(o.saguaro_request(xt, xd, T, 1, us)["tokens"][j])

    law = defaultdict(float)
    for v, a, b in step_law(f):
        law[v] += b - a
    return law


def pin_saguaro_toy_topk(o):
    """Residual top-3 on the toy tables: [0,.6,.2,.2,0,0,0] -> token 1 first,
    then {2, 3}; [0,.5,.25,0,0,0,.25] -> token 1, then {2, 6}.  The two equal
    values are equal only in exact arithmetic (the logits are ln of the
    tables), so their order is left to rounding and both slots must be flagged
    as ambiguous.  (Exact ties going to the lower index is pinned by
    pin_topk against numpy's stable argsort.)"""
    d0, d1, t0, t1 = toy_tables()
    for p, q, rest, vals in [(d0, t0, {2, 3}, [.6, .2, .2]), (d1, t1, {2, 6}, [.5, .25, .25])]:
        xt = np.log(np.stack([q, q]))
        xd = np.log(p)[None]
        r = o.saguaro_request(xt, xd, 1.0, 3, [0.3, 0.3], stats=True)
        top = list(r["topk"][0])
        assert top[0] == 1 and set(top[1:]) == rest, top
        assert r["topk_flag"][0] & 0b110 == 0b110 and r["topk_flag"][0] & 1 == 0
        assert abs(r["stats"][0, 2] - (1 - np.minimum(p, q).sum())) < 1e-9
        assert abs(r["stats"][0, 5] - vals[0]) < 1e-9 and abs(r["stats"][0, 6] - vals[2]) < 1e-9


def pin_saguaro_bonus_position(o):
    """At j = gamma the residual and p_D are both q, and sqrt(q * q) = q: the
    Saguaro sample at the bonus position follows the target exactly."""
    from scipy.special import softmax
    rng = np.random.Generator(np.random.PCG64(15))
    V, T = 6, 0.9
    xt = rng.normal(0, 1.0, (2, V))
    xd = rng.normal(0, 1.0, (1, V))
    law = sag_token_law(o, xt, xd, T, 1)
    q = softmax(xt[1] / T)
    assert np.allclose([law.get(v, 0.0) for v in range(V)], q, atol=1e-9)
    r = o.saguaro_request(xt, xd, T, 3, [0.5, 0.5])
    assert list(r["topk"][1]) == list(np.argsort(-q, kind="stable")[:3])


def pin_saguaro_disjoint_supports(o):
    """Target and draft with disjoint supports: the residual is q (S = 1), p_D
    vanishes on q's support and the residual vanishes on p_D's, so only the
    clamp survives: p_saguaro = sqrt(p_D) / sum sqrt(p_D) on p_D's support."""
    from scipy.special import softmax
    ninf = -np.inf
    zt = np.array([0.3, -0.2, 0.9, ninf, ninf, ninf])
    zd = np.array([ninf, ninf, ninf, 0.5, -1.0, 0.1])
    xt = np.stack([zt, zt])
    xd = zd[None]
    T = 1.0
    law = sag_token_law(o, xt, xd, T, 0)
    pD = softmax(zd / T)
    want = np.sqrt(pD) / np.sqrt(pD).sum()
    assert np.allclose([law.get(v, 0.0) for v in range(6)], want, atol=1e-9)
    r = o.saguaro_request(xt, xd, T, 2, [0.5, 0.5], stats=True)
    assert list(r["topk"][0]) == [2, 0]
    assert abs(r["stats"][0, 2] - 1.0) < 1e-12


def pin_saguaro_equal_distributions(o):
    """q == p: no residual mass, the residual falls back to q, and
    sqrt(p * q) = q: the Saguaro sample follows the target."""
    from scipy.special import softmax
    rng = np.random.Generator(np.random.PCG64(16))
    V, T = 5, 1.3
    z = rng.normal(0, 1.0, V)
    xt = np.stack([z, z])
    xd = z[None]
    law = sag_token_law(o, xt, xd, T, 0)
    assert np.allclose([law.get(v, 0.0) for v in range(V)], softmax(z / T), atol=1e-9)


def pin_cache_hit_rate(o):
    """A round hits the Saguaro cache when its correction / bonus token is
    among the top-k predicted for its acceptance length n.  Over the round's
    uniforms (exact law by enumeration) the hit probability must equal the
    closed form sum_n P(N = n) * (mass of r_n on its top-k), with
    P(N = n) = a_0 ... a_{n-1} (1 - a_n), a_i = min(1, q_i(x_i) / p_i(x_i)),
    r_n the normalised residual (q_gamma at n = gamma): the accept rule and
    residual law of the verification section, composed with the cache rule."""
    from scipy.special import softmax
    rng = np.random.Generator(np.random.PCG64(21))
    V, g, T, k = 6, 2, 0.9, 2
    xt = rng.normal(0, 1.0, (g + 1, V))
    xd = rng.normal(0, 1.0, (g, V))
    tok = np.array([int(np.argmax(xd[0])), int(np.argsort(xd[1])[-2])], np.int32)
    top = o.saguaro_request(xt, xd, T, k, np.full(g + 1, 0.5))["topk"]
    law = request_law(o, xt, xd, T, tok)
    p_hit = 0.0
    for out, pr in law.items():  # out: x_0 .. x_{n-1}, the correction / bonus at n, then -1
        n = len(emitted(out)) - 1
        row = np.array([out], np.int32)
        hit, count = o.cache_check(top[None], row, np.array([n], np.int32))
        assert count == (1 if hit[0] >= 0 else 0)
        if hit[0] >= 0:
            assert top[n, hit[0]] == out[n]
            p_hit += pr
    q = softmax(xt / T, axis=1)
    p = softmax(xd / T, axis=1)
    a = [min(1.0, q[i, tok[i]] / p[i, tok[i]]) for i in range(g)]
    closed = 0.0
    for n in range(g + 1):
        r = q[g] if n == g else np.maximum(q[n] - p[n], 0.0)
        r = r / r.sum()
        mass = r[np.argsort(-r, kind="stable")[:k]].sum()
        pn = np.prod(a[:n]) * (1.0 - a[n] if n < g else 1.0)
        closed += pn * mass
    assert abs(p_hit - closed) < 1e-9, (p_hit, closed)
    # an error outcome (n = -1) never hits
    hit, count = o.cache_check(top[None], np.full((1, g + 1), -1, np.int32), np.array([-1], np.int32))
    assert hit[0] == -1 and count == 0


def pin_draft_topk(o):
    """The bonus predictor of the SSD notes (section 3.1) takes the top-k of
    the draft logits.  On the verification blog's toy tables (draft after
    token 0: .55 .15 .10 .07 .06 .04 .03; after another token: .30 .20 .15
    .12 .10 .08 .05) the draft top-3 is [0, 1, 2] in both rows and the
    reported values are the printed probabilities.  On random logits with
    planted ties it equals numpy's stable argsort of the negated logits (the
    draft row for j < gamma, the target row at j = gamma), and the Saguaro
    draw does not depend on where the top-k comes from."""
    d0, d1, t0, t1 = toy_tables()
    for p, q in [(d0, t0), (d1, t1)]:
        xt = np.log(np.stack([q, q]))
        xd = np.log(p)[None]
        r = o.saguaro_request(xt, xd, 1.0, 3, [0.3, 0.3], stats=True, source="draft")
        assert list(r["topk"][0]) == [0, 1, 2], r["topk"][0]
        assert abs(r["stats"][0, 5] - p[0]) < 1e-12 and abs(r["stats"][0, 6] - p[2]) < 1e-12
        assert list(r["topk"][1]) == list(np.argsort(-q, kind="stable")[:3])
        assert r["topk_flag"][0] == 0
    rng = np.random.Generator(np.random.PCG64(23))
    V, g, k, T = 40, 3, 5, 0.7
    xt = np.round(rng.normal(0, 1.0, (g + 1, V)), 1)
    xd = np.round(rng.normal(0, 1.0, (g, V)), 1)
    u = rng.random(g + 1)
    r = o.saguaro_request(xt, xd, T, k, u, source="draft")
    for j in range(g + 1):
        row = xd[j] if j < g else xt[g]
        assert list(r["topk"][j]) == list(np.argsort(-row, kind="stable")[:k]), j
    r0 = o.saguaro_request(xt, xd, T, k, u, source="residual")
    assert list(r["tokens"]) == list(r0["tokens"])


def pin_saguaro_draft_lossless(o):
    """Draft tokens sampled from the Saguaro distribution p' of their position
    (the SSD notes, section 3.2) and verified with p' in p's place: the first
    emitted token follows q exactly, averaged over x_0 ~ p' (the verification
    blog's acceptance theorem holds for any draft distribution; the SSD notes'
    section 5.1 reads SSD as standard SD under Saguaro sampling).  The same
    tokens verified against the plain p give a different law."""
    from scipy.special import softmax
    rng = np.random.Generator(np.random.PCG64(25))
    V, T = 5, 0.9
    for g in (1, 2):
        xt = rng.normal(0, 1.0, (g + 1, V))
        xd = rng.normal(0, 1.0, (g, V))
        q0 = softmax(xt[0] / T)
        # the Saguaro distribution of position 0, as the oracle's Saguaro step
        # defines it (its clamp order is pinned by pin_saguaro_clamp_order)
        _, psag = o.saguaro_position(xt[0], xd[0], T)
        marg, marg_plain = np.zeros(V), np.zeros(V)
        for x0 in range(V):
            tok = [x0] + [int(np.argmax(xd[i])) for i in range(1, g)]
            for out, pr in request_law(o, xt, xd, T, tok, draft_dist="saguaro").items():
                marg[out[0]] += psag[x0] * pr
            for out, pr in request_law(o, xt, xd, T, tok).items():
                marg_plain[out[0]] += psag[x0] * pr
        assert np.allclose(marg, q0, atol=1e-9), (marg, q0)
        assert np.abs(marg_plain - q0).max() > 1e-3


def pin_top_p(o):
    """Top-p composed with verification (the verification blog's closing
    remark and its section on matching sampling parameters: speculative
    decoding stacks on temperature and top-p when both sides truncate the same
    way).  On the printed toy tables at top_p = 0.75 the target after token 0
    (.50 .18 .11 .08 ...) keeps {0, 1, 2} (mass .79) and the draft (.55 .15
    .10 ...) keeps {0, 1, 2} (.80); at 0.8 the target keeps {0, 1, 2, 3}.  With
    x_0 drawn from the truncated draft, the first emitted token follows the
    truncated target exactly.  Tokens tied with the last one needed are kept;
    top_p = 1 changes nothing."""
    d0, d1, t0, t1 = toy_tables()
    qP, amb = o.nucleus(np.log(t0), t0, 0.75)
    assert not amb and np.allclose(qP, np.r_[t0[:3] / t0[:3].sum(), np.zeros(4)], atol=1e-12)
    pP, amb = o.nucleus(np.log(d0), d0, 0.75)
    assert not amb and np.allclose(pP, np.r_[d0[:3] / d0[:3].sum(), np.zeros(4)], atol=1e-12)
    q8, _ = o.nucleus(np.log(t0), t0, 0.8)
    assert np.count_nonzero(q8) == 4
    # first emitted token of a round, x_0 ~ truncated draft: the truncated target
    xt = np.log(np.stack([t0, t1]))
    xd = np.log(d0)[None]
    marg = np.zeros(7)
    for x0 in range(7):
        if pP[x0] == 0:
            continue
        for out, pr in request_law(o, xt, xd, 1.0, [x0], top_p=0.75).items():
            marg[out[0]] += pP[x0] * pr
    assert np.allclose(marg, qP, atol=1e-9), (marg, qP)
    # ties at the boundary: logits 2, 1, 1, 1, 0 -- reaching 0.5 needs one of the
    # three tied tokens, so all three are kept
    x = np.array([2.0, 1.0, 1.0, 1.0, 0.0])
    from scipy.special import softmax
    pr = softmax(x)
    kept, _ = o.nucleus(x, pr, 0.5)
    assert list(np.nonzero(kept)[0]) == [0, 1, 2, 3]
    # top_p = 1: the plain verification
    rng = np.random.Generator(np.random.PCG64(27))
    xt = rng.normal(0, 1.0, (3, 9))
    xd = rng.normal(0, 1.0, (2, 9))
    for seed in range(20):
        u = np.random.default_rng(seed).random((2, 3))
        a = o.verify_request(xt, xd, 0.8, [1, 4], u[0], u[1])
        b = o.verify_request(xt, xd, 0.8, [1, 4], u[0], u[1], top_p=1.0)
        assert list(a["out"]) == list(b["out"])


def pin_saguaro_clamp_order(o):
    """The SSD notes (section 3.2) clamp the residual once it is a probability
    vector -- r = (q - p)+ / S, then max(r, 1e-8) -- and renormalise the mix.
    A row whose residual has one positive entry makes the order visible: with
    a uniform draft p = 1/V and q moving mass S from every other token onto
    token 0, r = (1, 0, ..., 0) whatever S is, so by hand
      p_saguaro(0) = sqrt(1/V) / (sqrt(1/V) + (V - 1) sqrt(1e-8 / V))
                   = 1 / (1 + (V - 1) 1e-4),
    Zs = sqrt(1/V) (1 + (V - 1) 1e-4), and every other token gets 1e-4 of
    token 0's probability -- the same for every S.  Clamping before the
    normalisation (max((q - p)+, 1e-8) / S) would give 1 / (1 + (V - 1) 1e-4 /
    sqrt(S)) instead."""
    V = 1001
    want0 = 1.0 / (1.0 + (V - 1) * 1e-4)
    want_zs = np.sqrt(1.0 / V) * (1.0 + (V - 1) * 1e-4)
    for S in (0.5, 0.2):
        q = np.full(V, 1.0 / V - S / (V - 1))
        q[0] = 1.0 / V + S
        xt = np.log(np.stack([q, q]))
        xd = np.zeros((1, V))
        r, ps, _, _, mass = o.saguaro_position(xt[0], xd[0], 1.0, full=True)
        assert abs(mass - S) < 1e-12, mass
        assert r[0] == 1.0 and np.all(r[1:] == 0.0)
        assert abs(ps[0] / want0 - 1) < 1e-12, (S, ps[0], want0)
        assert np.allclose(ps[1:], 1e-4 * ps[0], rtol=1e-12, atol=0)
        res = o.saguaro_request(xt, xd, 1.0, 1, [0.5, 0.5], stats=True)
        assert res["tokens"][0] == 0
        assert abs(res["stats"][0, 3] / want_zs - 1) < 1e-12 and abs(res["stats"][0, 4] / want0 - 1) < 1e-12
        # the law's first step: token 0 owns [0, p_saguaro(0))
        assert o.saguaro_request(xt, xd, 1.0, 1, [want0 - 1e-9, 0.5])["tokens"][0] == 0
        assert o.saguaro_request(xt, xd, 1.0, 1, [want0 + 1e-9, 0.5])["tokens"][0] == 1


def pin_draw_row(o):
    """A token's CDF interval in a request's draw row, and the row's flag mass.
    Closed forms: a uniform row of V tokens gives token t the interval
    [t/V, (t+1)/V) and flag mass V * min(1/V, 2 band); a residual row of mass
    below the band flags every draw (mass 1).  Against the pinned decision
    function: the token the oracle draws for a uniform u owns an interval
    holding u, the intervals tile [0, 1), and the share of uniforms the
    oracle flags matches the mass (binomial, 5 sigma)."""
    z = np.zeros((2, 50))
    for V, band, fm_want in [(50, 1e-3, 50 * 2e-3), (1000, 1e-3, 1.0)]:
        xt = np.zeros((2, V))
        xd = np.zeros((1, V))
        for t in (0, 7, V - 1):
            lo, hi, fm = o.draw_row(xt, xd, 1.0, [0], 1, t, band=band)
            assert abs(lo - t / V) < 1e-14 and abs(hi - (t + 1) / V) < 1e-14
            assert abs(fm - fm_want) < 1e-12, (V, fm)
    rng = np.random.Generator(np.random.PCG64(31))
    xd = rng.normal(0, 1.0, (1, 60))
    xt = np.stack([xd[0] + 1e-10 * rng.normal(size=60), xd[0]])
    assert o.draw_row(xt, xd, 1.0, [3], 0, 5)[2] == 1.0
    V, g = 40, 2
    xt = rng.normal(0, 1.2, (g + 1, V))
    xd = rng.normal(0, 1.2, (g, V))
    p0 = np.exp(xd[0] - xd[0].max())
    q0 = np.exp(xt[0] - xt[0].max())
    tok = [int(np.argmax(p0 / p0.sum() - q0 / q0.sum())), 3]  # q(x) < p(x): rejected at u = 1 - 2^-24
    for u in np.concatenate([rng.random(40), [0.0, 1 - 2**-24]]):
        out = o.verify_request(xt, xd, 1.0, tok, [1 - 2**-24, 0.5], [u, 0.5, 0.5])["out"]
        lo, hi, _ = o.draw_row(xt, xd, 1.0, tok, 0, int(out[0]))
        assert lo <= u < hi, (u, lo, hi)
        out = o.verify_request(xt, xd, 1.0, tok, [0.0, 0.0], [0.5, 0.5, u])["out"]
        lo, hi, _ = o.draw_row(xt, xd, 1.0, tok, g, int(out[g]))
        assert lo <= u < hi, (u, lo, hi)
    edges = [o.draw_row(xt, xd, 1.0, tok, 0, t)[:2] for t in range(V)]
    assert edges[0][0] == 0.0 and abs(edges[-1][1] - 1.0) < 1e-12
    assert all(edges[t][1] == edges[t + 1][0] for t in range(V - 1))
    band = 4e-3
    fm = o.draw_row(xt, xd, 1.0, tok, 0, 0, band=band)[2]
    n, flagged = 4000, 0
    for u in rng.random(n):
        r = o.verify_request(xt, xd, 1.0, tok, [1 - 2**-24, 0.5], [u, 0.5, 0.5], band=band)
        flagged += r["flag_pos"] == 0 and r["flag_kind"] == 1
    sd = np.sqrt(n * fm * (1 - fm))
    assert abs(flagged - n * fm) <= 5 * sd + 1, (flagged, n * fm)


ALL_PINS = [
    pin_philox_vs_triton, pin_uniform_mapping, pin_uniform_statistics, pin_softmax, pin_argmax,
    pin_topk, pin_choice, pin_toy_closed_forms, pin_losslessness_toy_chain,
    pin_losslessness_random, pin_greedy, pin_low_temperature_limit, pin_expected_tokens,
    pin_toy_kl, pin_saguaro_toy_topk, pin_saguaro_bonus_position,
    pin_saguaro_disjoint_supports, pin_saguaro_equal_distributions, pin_cache_hit_rate, pin_draft_topk,
    pin_saguaro_draft_lossless, pin_top_p, pin_saguaro_clamp_order, pin_draw_row,
]
