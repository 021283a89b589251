"""Pins for the CPU oracle: facts the pages and the mathematics fix, checked
without any GPU and without the CUDA library.

* exact induced law on tiny vocabularies (the rule is exact in distribution:
  "Decodificación Especulativa y EAGLE", section "La Regla de Exactitud");
* chi-square over 10^6 trials and the TV < 0.01 exercise (same lesson,
  section "Ejercicios");
* the closed form for expected tokens and its printed value 3.36 (section
  "Aceleración Esperada", fixture tests/golden/expected_tokens.txt);
* the greedy rule (section "Caso codicioso") against numpy's argmax;
* the n+1 bound ("Accelerating Sonar through speculation", section
  "Decodificación especulativa") and the step-shape statements of section
  "El Concepto" (fixture tests/golden/speculative_step_shape.txt);
* special cases: p = q, disjoint supports, vanishing temperature.

The model distributions in these tests come from scipy.special.softmax, not
from the oracle's own code.
"""

import itertools
import os

import numpy as np
import pytest
from scipy import stats
from scipy.special import softmax

import oracle
from speculative_decoding_verify_sample_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _dist(z, T):
    return softmax(np.asarray(z, np.float64) / float(np.float32(T)))


def _batch(zp, zq, x, n, T, u, ur, dtype="f32"):
    """Replicate one set of logits over a batch of requests."""
    B = len(x)
    K = zq.shape[0]
    V = zp.shape[1]
    tgt = np.ascontiguousarray(np.broadcast_to(zp, (B, K + 1, V)))
    drf = np.ascontiguousarray(np.broadcast_to(zq, (B, K, V)))
    return dict(B=B, K=K, V=V, dtype=dtype, target=tgt, draft=drf,
                draft_tokens=np.asarray(x, np.int32).reshape(B, K),
                draft_len=np.full(B, n, np.int32), temperature=np.full(B, T, np.float32),
                uniforms=np.asarray(u, np.float32).reshape(B, K + 1),
                uniforms_resample=np.asarray(ur, np.float32).reshape(B))


def _intervals(edges):
    pts = np.unique(np.concatenate([[0.0], np.clip(edges, 0.0, 1.0), [1.0]]))
    lo, hi = pts[:-1], pts[1:]
    keep = hi - lo > 0
    lo, hi = lo[keep], hi[keep]
    assert np.all(hi - lo > 1e-5), "edges too close for fp32 midpoints; choose another seed"
    return (lo + hi) / 2, hi - lo


def _cdf_edges(w):
    c = np.cumsum(w) / np.sum(w)
    return c[:-1]


def induced_law(zp, zq, n, T, dtype="f32"):
    """Exact law of (accepted_len, emitted tokens) of the oracle for drafts
    x_t ~ q_t: the oracle is evaluated at the midpoint of every interval on
    which its output is constant in each uniform, weighted by the interval's
    length and by prod_t q_t(x_t)."""
    K, V = zq.shape
    zpf = synth.as_f32(zp, dtype)
    zqf = synth.as_f32(zq, dtype)
    p = [_dist(zpf[t], T) for t in range(n + 1)]
    q = [_dist(zqf[t], T) for t in range(n)]
    res_edges = np.concatenate([_cdf_edges(np.maximum(p[t] - q[t], 0.0)) for t in range(n)])
    ur_mid, ur_len = _intervals(res_edges)
    ub_mid, ub_len = _intervals(_cdf_edges(p[n]))
    xs, us, urs, wts = [], [], [], []
    for x in itertools.product(range(V), repeat=n):
        wx = np.prod([q[t][x[t]] for t in range(n)])
        if wx == 0:
            continue
        for pattern in itertools.product((True, False), repeat=n):
            ut, lt = [], 1.0
            for t in range(n):
                ratio = min(p[t][x[t]] / q[t][x[t]], 1.0)
                a, b = (0.0, ratio) if pattern[t] else (ratio, 1.0)
                if b - a <= 0:
                    lt = 0.0
                    break
                assert b - a > 1e-5
                ut.append((a + b) / 2)
                lt *= b - a
            if lt == 0.0:
                continue
            for um, ul in zip(ub_mid, ub_len):
                for rm, rl in zip(ur_mid, ur_len):
                    u = np.zeros(K + 1)
                    u[:n] = ut
                    u[n] = um
                    xs.append(list(x) + [0] * (K - n))
                    us.append(u)
                    urs.append(rm)
                    wts.append(wx * lt * ul * rl)
    inp = _batch(zp, zq, xs, n, T, us, urs, dtype)
    acc, out, flags = oracle.verify_sample(inp)
    assert np.all(flags & oracle.BAD_INPUT == 0)
    law = {}
    for j, row, w in zip(acc, out, wts):
        key = (int(j), tuple(int(v) for v in row[: j + 1]))
        law[key] = law.get(key, 0.0) + w
    return law, p, q


ENUM_CASES = [
    # (seed, V, K, n, T, dtype)
    (11, 4, 2, 2, 1.0, "f32"),
    (12, 3, 3, 3, 0.7, "f32"),
    (13, 6, 2, 2, 1.3, "f32"),
    (14, 4, 3, 2, 1.0, "f32"),      # ragged: n < K, bonus from row n
    (15, 5, 2, 2, 0.5, "bf16"),
    (16, 8, 1, 1, 1.0, "f32"),
]


@pytest.mark.parametrize("seed,V,K,n,T,dtype", ENUM_CASES)
def test_exact_enumeration_matches_target_law(seed, V, K, n, T, dtype):
    rng = np.random.default_rng(seed)
    zq = (1.5 * rng.standard_normal((K, V))).astype(np.float32)
    zp = (1.5 * rng.standard_normal((K + 1, V))).astype(np.float32)
    if dtype == "bf16":
        zq, zp = synth.bf16_bits(zq), synth.bf16_bits(zp)
    law, p, q = induced_law(zp, zq, n, T, dtype)
    assert abs(sum(law.values()) - 1.0) < 1e-12
    alpha = [np.minimum(p[t], q[t]).sum() for t in range(n)]
    reach = np.cumprod([1.0] + alpha)            # P(j >= t)
    for t in range(n + 1):
        got_reach = sum(w for (j, _), w in law.items() if j >= t)
        assert abs(got_reach - reach[t]) < 1e-12, (t, got_reach, reach[t])
        # the token emitted at position t, jointly with reaching t, is p_t
        for v in range(V):
            mass = sum(w for (j, toks), w in law.items() if j >= t and toks[t] == v)
            assert abs(mass - reach[t] * p[t][v]) < 1e-12, (t, v, mass, reach[t] * p[t][v])


def test_exact_enumeration_target_zero_probability_token():
    """p(x) = 0 for some drafted x (target logit -inf): those drafts are
    always rejected and the law is still p."""
    rng = np.random.default_rng(21)
    V, K, n = 5, 2, 2
    zq = rng.standard_normal((K, V)).astype(np.float32)
    zp = rng.standard_normal((K + 1, V)).astype(np.float32)
    zp[0, 1] = -np.inf
    zp[1, 3] = -np.inf
    law, p, q = induced_law(zp, zq, n, 1.0)
    assert abs(sum(law.values()) - 1.0) < 1e-12
    for v in range(V):
        mass = sum(w for (_, toks), w in law.items() if toks[0] == v)
        assert abs(mass - p[0][v]) < 1e-12
    assert sum(w for (_, toks), w in law.items() if toks[0] == 1) == 0.0


def _chi2_trials(seed, V, K, T, trials, chunk=125_000):
    rng = np.random.default_rng(seed)
    zq = (1.2 * rng.standard_normal((K, V))).astype(np.float32)
    zp = (zq[np.r_[0:K, K - 1]] + 0.8 * rng.standard_normal((K + 1, V))).astype(np.float32)
    p = [_dist(zp[t], T) for t in range(K + 1)]
    q = [_dist(zq[t], T) for t in range(K)]
    first = np.zeros(V)
    lens = np.zeros(K + 1)
    for _ in range(trials // chunk):
        x = np.stack([rng.choice(V, size=chunk, p=q[t]) for t in range(K)], axis=1)
        u = synth.uniforms24(rng, (chunk, K + 1))
        ur = synth.uniforms24(rng, (chunk,))
        acc, out, flags = oracle.verify_sample(_batch(zp, zq, x, K, T, u, ur), nthreads=4)
        assert np.all(flags & oracle.BAD_INPUT == 0)
        first += np.bincount(out[:, 0], minlength=V)
        lens += np.bincount(acc, minlength=K + 1)
    alpha = np.array([np.minimum(p[t], q[t]).sum() for t in range(K)])
    reach = np.cumprod(np.r_[1.0, alpha])
    law_len = np.r_[reach[:K] * (1.0 - alpha), reach[K]]
    return first, lens, p[0], law_len


def test_chi_square_million_trials():
    trials = 1_000_000
    first, lens, p0, law_len = _chi2_trials(31, 16, 4, 1.0, trials)
    assert first.sum() == trials
    c1 = stats.chisquare(first, p0 * trials)
    c2 = stats.chisquare(lens, law_len * trials)
    assert c1.pvalue > 1e-3, c1
    assert c2.pvalue > 1e-3, c2
    # the lesson's exercise: total variation to plain sampling from p below 0.01
    assert 0.5 * np.abs(first / trials - p0).sum() < 0.01


def test_chi_square_detects_wrong_law():
    """The same statistic rejects a law that differs from p by a few percent,
    so the pass above is not vacuous."""
    trials = 1_000_000
    first, _, p0, _ = _chi2_trials(31, 16, 4, 1.0, trials)
    wrong = 0.97 * p0 + 0.03 * np.roll(p0, 1)
    assert stats.chisquare(first, wrong * trials).pvalue < 1e-6


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def _closed_form(alpha, K):
    return (1.0 - alpha ** (K + 1)) / (1.0 - alpha)


def test_closed_form_printed_value():
    (alpha, K, printed, dec), = _golden_rows("expected_tokens.txt")
    alpha, K, printed, dec = float(alpha), int(K), float(printed), int(dec)
    # the formula, summed term by term (1 + a + ... + a^K), against the print
    series = sum(alpha ** i for i in range(K + 1))
    assert round(series, dec) == printed
    assert abs(series - _closed_form(alpha, K)) < 1e-12


def _expected_tokens_trial(alpha, K, n_req, V=64, seed=41, draft_len=None):
    rng = np.random.default_rng(seed)
    logp, logq = synth.constant_overlap_rows(rng, n_req * (K + 1), V, np.full(n_req * (K + 1), alpha))
    tgt = logp.reshape(n_req, K + 1, V)
    drf = np.ascontiguousarray(logq.reshape(n_req, K + 1, V)[:, :K])
    T = np.ones(n_req, np.float32)
    toks = synth.gumbel_draw(rng, drf.reshape(n_req * K, V), np.repeat(T, K)).reshape(n_req, K)
    inp = dict(B=n_req, K=K, V=V, dtype="f32", target=tgt, draft=drf, draft_tokens=toks,
               draft_len=draft_len, temperature=T,
               uniforms=synth.uniforms24(rng, (n_req, K + 1)),
               uniforms_resample=synth.uniforms24(rng, (n_req,)))
    acc, out, flags = oracle.verify_sample(inp, nthreads=4)
    return acc, out, inp


def test_closed_form_expected_tokens_constant_overlap():
    (alpha, K, printed, _), = _golden_rows("expected_tokens.txt")
    alpha, K, printed = float(alpha), int(K), float(printed)
    n_req = 40_000
    acc, _, _ = _expected_tokens_trial(alpha, K, n_req)
    emitted = acc + 1.0
    mean, se = emitted.mean(), emitted.std() / np.sqrt(n_req)
    assert abs(mean - _closed_form(alpha, K)) < 4 * se, (mean, se)
    assert abs(mean - printed) < 4 * se + 0.005
    # per-position acceptance equals the constructed overlap
    reached = acc[:, None] >= np.arange(K)[None, :]
    accepted = acc[:, None] > np.arange(K)[None, :]
    rate = accepted.sum(0) / reached.sum(0)
    assert np.all(np.abs(rate - alpha) < 4 * np.sqrt(alpha * (1 - alpha) / reached.sum(0)))


@pytest.mark.parametrize("alpha", [0.5, 0.95])
def test_closed_form_ragged_draft_lengths(alpha):
    K, n_req = 8, 24_000
    rng = np.random.default_rng(43)
    n = rng.integers(1, K + 1, size=n_req).astype(np.int32)
    acc, _, _ = _expected_tokens_trial(alpha, K, n_req, V=32, seed=44, draft_len=n)
    want = np.mean([_closed_form(alpha, int(k)) for k in n])
    emitted = acc + 1.0
    assert abs(emitted.mean() - want) < 4 * emitted.std() / np.sqrt(n_req)


def test_greedy_rule_against_numpy_argmax_with_ties():
    rng = np.random.default_rng(51)
    B, K, V = 300, 4, 37
    # values from a small set: exact ties at the maximum are common
    zp = rng.integers(-3, 4, size=(B, K + 1, V)).astype(np.float32) * 0.5
    g = np.argmax(zp, axis=2)            # numpy: first occurrence = lowest index
    hit = rng.random((B, K)) < 0.6
    x = np.where(hit, g[:, :K], rng.integers(0, V, size=(B, K))).astype(np.int32)
    n = rng.integers(1, K + 1, size=B).astype(np.int32)
    for dtype in ("f32", "bf16"):
        tgt = synth.bf16_bits(zp) if dtype == "bf16" else zp
        inp = dict(B=B, K=K, V=V, dtype=dtype, target=tgt, draft=None, draft_tokens=x,
                   draft_len=n, temperature=np.zeros(B, np.float32),
                   uniforms=synth.uniforms24(rng, (B, K + 1)),
                   uniforms_resample=synth.uniforms24(rng, (B,)))
        acc, out, flags = oracle.verify_sample(inp)
        assert np.all(flags == 0)
        for b in range(B):
            j = next((t for t in range(n[b]) if g[b, t] != x[b, t]), n[b])
            want = list(x[b, :j]) + [g[b, j]] + [-1] * (K - j)
            assert acc[b] == j
            assert list(out[b]) == want


def test_greedy_tie_goes_to_lowest_index():
    V, K = 10, 2
    zp = np.zeros((1, K + 1, V), np.float32)
    zp[0, 0, [3, 7]] = 5.0
    zp[0, 1, [0, 9]] = 2.0
    zp[0, 2, [4, 5, 6]] = 1.0
    x = np.array([[3, 9]], np.int32)
    inp = dict(B=1, K=K, V=V, dtype="f32", target=zp, draft=None, draft_tokens=x, draft_len=None,
               temperature=np.zeros(1, np.float32), uniforms=np.zeros((1, K + 1), np.float32),
               uniforms_resample=np.zeros(1, np.float32))
    acc, out, _ = oracle.verify_sample(inp)
    assert acc[0] == 1 and list(out[0]) == [3, 0, -1]
    x[0, 1] = 0
    acc, out, _ = oracle.verify_sample(inp)
    assert acc[0] == 2 and list(out[0]) == [3, 0, 4]


def _check_bound(inp, acc, out):
    K = inp["K"]
    n = np.full(inp["B"], K) if inp["draft_len"] is None else inp["draft_len"]
    for b in range(inp["B"]):
        j = acc[b]
        assert 0 <= j <= n[b]
        assert list(out[b, :j]) == list(inp["draft_tokens"][b, :j])
        assert 0 <= out[b, j] < inp["V"]
        assert np.all(out[b, j + 1:] == -1)
        assert j + 1 <= n[b] + 1


@pytest.mark.parametrize("name", ["tiny", "tiny_greedy"])
def test_n_plus_one_bound_named(name):
    inp = synth.make_inputs(name)
    acc, out, _ = oracle.verify_sample(inp)
    _check_bound(inp, acc, out)


def test_n_plus_one_bound_random_mixed():
    inp = synth.random_case(61, B=200, K=6, V=50, temperature=0.9, draft_len="random",
                            greedy_frac=0.3)
    acc, out, flags = oracle.verify_sample(inp)
    assert np.all(flags & oracle.BAD_INPUT == 0)
    _check_bound(inp, acc, out)


def test_step_shape_statements():
    rows = {r[0]: (int(r[1]), int(r[2])) for r in _golden_rows("speculative_step_shape.txt")}
    K, want = rows["perfect_draft"]
    rng = np.random.default_rng(71)
    V, B = 40, 50
    z = rng.standard_normal((B, K + 1, V)).astype(np.float32)
    inp = dict(B=B, K=K, V=V, dtype="f32", target=z, draft=np.ascontiguousarray(z[:, :K]),
               draft_tokens=rng.integers(0, V, size=(B, K)).astype(np.int32), draft_len=None,
               temperature=np.full(B, 0.8, np.float32),
               uniforms=synth.uniforms24(rng, (B, K + 1)),
               uniforms_resample=synth.uniforms24(rng, (B,)))
    acc, out, _ = oracle.verify_sample(inp)
    # p = q: p(x)/q(x) = 1 > u for every draft, so all K are kept plus a bonus
    assert np.all(acc + 1 == want)
    K, want = rows["first_position_wrong"]
    z2 = np.full((B, K + 1, V), -np.inf, np.float32)
    zq = np.full((B, K, V), -np.inf, np.float32)
    z2[:, :, : V // 2] = rng.standard_normal((B, K + 1, V // 2))
    zq[:, :, V // 2:] = rng.standard_normal((B, K, V - V // 2))
    x = rng.integers(V // 2, V, size=(B, K)).astype(np.int32)
    inp.update(target=z2, draft=zq, draft_tokens=x)
    acc, out, flags = oracle.verify_sample(inp)
    # disjoint supports: x ~ q has p(x) = 0, rejected at once; residual = p
    assert np.all(acc + 1 == want)
    assert np.all(out[:, 0] < V // 2)


def test_vanishing_temperature_equals_greedy():
    rng = np.random.default_rng(81)
    B, K, V = 100, 3, 30
    # a clear maximum in every row: top gap >= 0.25
    zp = rng.standard_normal((B, K + 1, V)).astype(np.float32)
    zq = zp[:, :K] + 0.7 * rng.standard_normal((B, K, V)).astype(np.float32)
    for z in (zp, zq):
        top = np.argmax(z, axis=2)
        bi, ti = np.meshgrid(np.arange(z.shape[0]), np.arange(z.shape[1]), indexing="ij")
        z[bi, ti, top] = z.max(axis=2) + 0.25
    x = np.argmax(zq, axis=2).astype(np.int32)         # what q draws at T -> 0
    base = dict(B=B, K=K, V=V, dtype="f32", target=zp, draft=np.ascontiguousarray(zq),
                draft_tokens=x, draft_len=None, uniforms=synth.uniforms24(rng, (B, K + 1)),
                uniforms_resample=synth.uniforms24(rng, (B,)))
    acc_s, out_s, _ = oracle.verify_sample(dict(base, temperature=np.full(B, 2e-3, np.float32)))
    acc_g, out_g, _ = oracle.verify_sample(dict(base, temperature=np.zeros(B, np.float32)))
    assert np.array_equal(acc_s, acc_g)
    assert np.array_equal(out_s, out_g)


def test_invalid_requests_are_flagged():
    inp = synth.random_case(91, B=6, K=3, V=20, temperature=1.0)
    inp["draft_len"] = np.array([3, 0, 4, 2, 3, 3], np.int32)
    inp["draft_tokens"][3, 1] = 20          # out of range, inside n = 2
    inp["draft_tokens"][0, 2] = 0
    inp["temperature"][4] = -1.0
    inp["uniforms_resample"][5] = 1.0
    acc, out, flags = oracle.verify_sample(inp)
    bad = (flags & oracle.BAD_INPUT) != 0
    assert list(bad) == [False, True, True, True, True, True]
    assert np.all(acc[bad] == -1) and np.all(out[bad] == -1)


def test_row_stats_probabilities_normalised():
    inp = synth.random_case(101, B=8, K=3, V=300, temperature=0.8, draft_len="random")
    info = oracle.row_stats(inp)
    zp = synth.as_f32(inp["target"], "f32")
    zq = synth.as_f32(inp["draft"], "f32")
    for b in range(inp["B"]):
        n = inp["draft_len"][b]
        for t in range(n):
            x = inp["draft_tokens"][b, t]
            p = _dist(zp[b, t], 0.8)
            q = _dist(zq[b, t], 0.8)
            assert abs(np.exp(info[b, t, 2]) - p[x]) <= 1e-12 * p[x] + 1e-300
            assert abs(np.exp(info[b, t, 5]) - q[x]) <= 1e-12 * q[x] + 1e-300
            assert abs(info[b, t, 6] - np.maximum(p - q, 0).sum()) < 1e-12
        assert np.all(np.isnan(info[b, n + 1:, 0]))


def test_sampled_request_with_unusable_row_is_flagged():
    """A sampled request whose needed rows include one without a finite
    maximum is invalid, even if the scan would stop before that row."""
    inp = synth.random_case(92, B=3, K=3, V=16, temperature=1.0)
    inp["target"][1, 3, :] = -np.inf        # the bonus row of request 1
    inp["draft"][2, 2, :] = -np.inf         # the last draft row of request 2
    acc, out, flags = oracle.verify_sample(inp)
    assert list((flags & oracle.BAD_INPUT) != 0) == [False, True, True]
    # greedy requests have an argmax on any row: no flag
    inp["temperature"][:] = 0.0
    acc, out, flags = oracle.verify_sample(inp)
    assert np.all(flags == 0)


# ---------------------------------------------------------------- near-tie flags
#
# The parity rules excuse a GPU/oracle mismatch only where the oracle sets a
# near-tie flag, so each flag is pinned here on constructed inputs whose
# ratio p(x)/q(x) and CDF edges are known (from scipy's softmax, not from the
# oracle): just inside a band the flag is set, just outside it is not.


def _one_request(zp, zq, x, u, ur, n=None):
    zp = np.asarray(zp, np.float32)
    zq = np.asarray(zq, np.float32)
    K = zq.shape[0]
    return dict(B=1, K=K, V=zp.shape[1], dtype="f32", target=zp[None].copy(),
                draft=zq[None].copy(), draft_tokens=np.asarray([x], np.int32),
                draft_len=None if n is None else np.asarray([n], np.int32),
                temperature=np.ones(1, np.float32),
                uniforms=np.asarray([u], np.float32), uniforms_resample=np.asarray([ur], np.float32))


def _f32(v):
    return float(np.float32(v))


@pytest.mark.parametrize("delta,flagged", [(-5e-5, True), (5e-5, True), (-9e-5, True),
                                           (9e-5, True), (-1.1e-4, False), (1.1e-4, False),
                                           (-2e-4, False), (2e-4, False)])
def test_tie_accept_band(delta, flagged):
    # p = (0.5, 0.5), q = (0.8, 0.2), x = 0: p(x)/q(x) = 0.625
    zp = np.log([[0.5, 0.5], [0.5, 0.5]])
    zq = np.log([[0.8, 0.2]])
    ratio = _dist(np.float32(zp[0]), 1.0)[0] / _dist(np.float32(zq[0]), 1.0)[0]
    u0 = _f32(ratio + delta)
    acc, out, flags = oracle.verify_sample(_one_request(zp, zq, [0], [u0, 0.25], 0.5))
    assert bool(flags[0] & oracle.TIE_ACCEPT) == flagged, (delta, flags[0])
    assert flags[0] & ~oracle.TIE_ACCEPT == 0          # no other flag on this input
    assert acc[0] == (1 if u0 < ratio else 0)          # strict u < p/q decides
    info = oracle.row_stats(_one_request(zp, zq, [0], [u0, 0.25], 0.5))
    assert bool(info[0, 0, 9]) == flagged


@pytest.mark.parametrize("edge_i,delta,flagged", [(1, -5e-5, True), (1, 5e-5, True),
                                                  (2, -9e-5, True), (0, 5e-5, True),
                                                  (1, -2e-4, False), (1, 2e-4, False),
                                                  (2, 1.2e-4, False), (0, -3e-4, False)])
def test_tie_cdf_band_bonus_draw(edge_i, delta, flagged):
    # p = q = (0.1, 0.2, 0.3, 0.4): the draft is always accepted and the bonus
    # token is drawn from p with uniforms[1]; CDF edges 0.1, 0.3, 0.6
    z = np.log([[0.1, 0.2, 0.3, 0.4]] * 2)
    edges = np.cumsum(_dist(np.float32(z[1]), 1.0))
    u1 = _f32(edges[edge_i] + delta)
    inp = _one_request(z, z[:1], [3], [0.5, u1], 0.5)
    acc, out, flags = oracle.verify_sample(inp)
    assert acc[0] == 1
    assert out[0, 1] == int(np.searchsorted(edges, u1, side="right"))
    assert bool(flags[0] & oracle.TIE_CDF) == flagged, (edge_i, delta, flags[0])
    assert flags[0] & ~oracle.TIE_CDF == 0
    info = oracle.row_stats(inp)
    assert info[0, 1, 7] == out[0, 1] and bool(info[0, 1, 8]) == flagged


def _small_residual_case():
    # q uniform over 4, p = (0.2505, 0.2505, 0.249, 0.25): (p - q)+ is about
    # (5e-4, 5e-4, 0, 0), W about 1e-3; x = 2 (p/q about 0.996) rejected by u = 0.999
    zp = np.log([[0.2505, 0.2505, 0.249, 0.25], [0.25] * 4])
    zq = np.zeros((1, 4))
    p = _dist(np.float32(zp[0]), 1.0)
    q = _dist(np.float32(zq[0]), 1.0)
    w = np.maximum(p - q, 0.0)
    return zp, zq, w


@pytest.mark.parametrize("offset,expect", [
    (6e-8, "tie_cdf"),        # |u'W - C_0| ~ 6e-11 < 1e-4 W
    (-6e-8, "tie_cdf"),
    (5e-3, "precision"),      # ~5e-6 of mass: inside 2e-5, outside 1e-4 W
    (-1.5e-2, "precision"),   # ~1.5e-5
    (3e-2, None),             # ~3e-5: outside both bands
    (-0.2, None),
    (0.3, None),
])
def test_residual_edge_bands_replace_small_mass_excuse(offset, expect):
    zp, zq, w = _small_residual_case()
    W = w.sum()
    assert 5e-4 < W < 2e-3                         # a residual far below 1 % of the mass
    c0 = w[0] / W                                  # the one interior edge, in u' units
    ur = _f32(c0 + offset)
    acc, out, flags = oracle.verify_sample(_one_request(zp, zq, [2], [0.999, 0.5], ur))
    assert acc[0] == 0
    assert out[0, 0] == (0 if ur * W < w[0] else 1)
    cdf = flags[0] & (oracle.TIE_CDF | oracle.PRECISION_BAND)
    want = {"tie_cdf": oracle.TIE_CDF, "precision": oracle.PRECISION_BAND, None: 0}[expect]
    assert cdf == want, (offset, flags[0])
    assert flags[0] & ~(oracle.TIE_CDF | oracle.PRECISION_BAND) == 0
    info = oracle.row_stats(_one_request(zp, zq, [2], [0.999, 0.5], ur))
    assert int(info[0, 0, 8]) == want and abs(info[0, 0, 6] - W) < 1e-15


@pytest.mark.parametrize("ur,token", [(0.3, 0), (0.7, 1)])
def test_zero_mass_residual_falls_back_to_p(ur, token):
    # q(x) = e^-40 / S and p(x) = e^-40.5 / S with S = 2 in both rows: in
    # double S_p == S_q, so p_i == q_i off x and p(x) < q(x); u = 0.9 rejects
    # x (p/q = e^-0.5) and the residual (p - q)+ is exactly zero
    zq = np.array([[0.0, 0.0, -40.0]])
    zp = np.array([[0.0, 0.0, -40.5], [0.0, 0.0, 0.0]])
    p = _dist(np.float32(zp[0]), 1.0)
    q = _dist(np.float32(zq[0]), 1.0)
    assert np.maximum(p - q, 0.0).sum() == 0.0 and p[2] < q[2]
    inp = _one_request(zp, zq, [2], [0.9, 0.5], ur)
    acc, out, flags = oracle.verify_sample(inp)
    assert acc[0] == 0 and out[0, 0] == token
    assert flags[0] & oracle.RES_FALLBACK
    info = oracle.row_stats(inp)
    assert info[0, 0, 6] == 0.0 and int(info[0, 0, 8]) & oracle.RES_FALLBACK
    assert info[0, 0, 7] == token


@pytest.mark.parametrize("u,token,tie", [(0.0, 1, False), (1 - 2 ** -24, 3, False),
                                         (0.5, 3, True), (0.25, 1, False), (0.75, 3, False)])
def test_inverse_cdf_never_emits_a_zero_weight_token(u, token, tie):
    # p = (0, 0.5, 0, 0.5, 0): leading, interior and trailing zero weights
    z = np.array([[-np.inf, 0.0, -np.inf, 0.0, -np.inf]] * 2)
    inp = _one_request(z, z[:1], [1], [0.5, u], 0.5)
    acc, out, flags = oracle.verify_sample(inp)
    assert acc[0] == 1 and out[0, 1] == token
    assert bool(flags[0] & oracle.TIE_CDF) == tie


def test_flags_agree_with_row_stats_on_random_requests():
    # the per-request flags are the union of the per-row flags of the rows the
    # scan evaluated: accept ties at rows 0..min(j, n-1), CDF flags at row j
    inp = synth.random_case(111, B=400, K=4, V=12, scale=1.0, noise=0.3, temperature=1.0,
                            draft_len="random")
    acc, out, flags = oracle.verify_sample(inp)
    info = oracle.row_stats(inp)
    n = inp["draft_len"]
    for b in range(inp["B"]):
        j = acc[b]
        evaluated = range(min(j, n[b] - 1) + 1)
        want_acc = any(info[b, t, 9] != 0 for t in evaluated)
        assert bool(flags[b] & oracle.TIE_ACCEPT) == want_acc, b
        assert flags[b] & (oracle.TIE_CDF | oracle.PRECISION_BAND | oracle.RES_FALLBACK) == \
            int(info[b, j, 8]), b
        assert out[b, j] == info[b, j, 7]
