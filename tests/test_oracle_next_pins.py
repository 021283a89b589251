"""Pins for the oracle's rows beyond the verification step itself: the
draft-side sampler, the one-hot (top-token) draft rule, greedy token-tree
verification, and the post-accept insert.  CPU only; the distributions come
from scipy.special.softmax, not from the oracle.

Pages (title, section):
* "Decodificación Especulativa y EAGLE": "La Configuración de Dos Modelos"
  and "Desarrolla" (the draft samples softmax(z/T)), "La Regla de
  Exactitud" (the rule for any q), "Caso codicioso" (argmax), "Verificación
  de Atención en Árvore" (token trees);
* "Accelerating Sonar through speculation": "Objetivo-Borrador" (the draft
  proposes its top token), "EAGLE" (trees), "Programación MTP para un solo
  token" (on-device insert of the next tokens).
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


def _mid_intervals(cdf):
    """Midpoints and lengths of the u-intervals [c_{i-1}, c_i) of a CDF."""
    pts = np.unique(np.concatenate([[0.0], np.clip(cdf, 0, 1), [1.0]]))
    lo, hi = pts[:-1], pts[1:]
    keep = hi - lo > 1e-9   # rounding slivers (a CDF sum of 1 - 1e-16): mass below 1e-8 in all
    return (lo[keep] + hi[keep]) / 2, hi[keep] - lo[keep]


# ---------------------------------------------------------------- draft-side sampler


@pytest.mark.parametrize("seed,V,T,dtype", [(1, 5, 1.0, "f32"), (2, 8, 0.6, "f32"),
                                            (3, 7, 1.4, "bf16"), (4, 3, 0.3, "f32")])
def test_sampler_exact_law_by_enumeration(seed, V, T, dtype):
    rng = np.random.default_rng(seed)
    z = (1.5 * rng.standard_normal(V)).astype(np.float32)
    if dtype == "bf16":
        z = synth.bf16_bits(z)
    p = _dist(synth.as_f32(z, dtype), T)
    mids, lens = _mid_intervals(np.cumsum(p)[:-1])
    R = len(mids)
    tok, flags = oracle.sample_draft(np.tile(z, (R, 1)), dtype, np.full(R, T, np.float32),
                                     mids.astype(np.float32))
    assert np.all(flags & oracle.BAD_INPUT == 0)
    law = np.zeros(V)
    np.add.at(law, tok, lens)
    assert np.max(np.abs(law - p)) < 1e-6   # fp32 midpoints: interval ends within 6e-8


def test_sampler_chi_square_million_draws():
    rng = np.random.default_rng(7)
    V, T, n = 32, 0.9, 1_000_000
    z = (1.2 * rng.standard_normal(V)).astype(np.float32)
    p = _dist(z, T)
    counts = np.zeros(V)
    for _ in range(4):
        m = n // 4
        tok, _ = oracle.sample_draft(np.broadcast_to(z, (m, V)), "f32", np.full(m, T, np.float32),
                                     synth.uniforms24(rng, (m,)), nthreads=4)
        counts += np.bincount(tok, minlength=V)
    assert stats.chisquare(counts, p * n).pvalue > 1e-3
    wrong = 0.97 * p + 0.03 * np.roll(p, 1)
    assert stats.chisquare(counts, wrong * n).pvalue < 1e-6


def test_sampler_greedy_is_lowest_argmax():
    rng = np.random.default_rng(9)
    R, V = 400, 23
    z = rng.integers(-3, 4, size=(R, V)).astype(np.float32)   # ties at the max are common
    tok, flags = oracle.sample_draft(z, "f32", np.zeros(R, np.float32), synth.uniforms24(rng, (R,)))
    assert np.array_equal(tok, np.argmax(z, axis=1)) and np.all(flags == 0)


def test_sampler_vanishing_temperature_is_argmax():
    rng = np.random.default_rng(10)
    R, V = 200, 40
    z = rng.standard_normal((R, V)).astype(np.float32)
    top = np.argmax(z, axis=1)
    z[np.arange(R), top] += 0.3
    tok, _ = oracle.sample_draft(z, "f32", np.full(R, 2e-3, np.float32), synth.uniforms24(rng, (R,)))
    assert np.array_equal(tok, top)


@pytest.mark.parametrize("u,token", [(0.0, 1), (0.49, 1), (0.51, 3), (1 - 2 ** -24, 3)])
def test_sampler_never_draws_zero_probability(u, token):
    z = np.array([[-np.inf, 0.0, -np.inf, 0.0, -np.inf]], np.float32)
    tok, _ = oracle.sample_draft(z, "f32", np.ones(1, np.float32), np.array([u], np.float32))
    assert tok[0] == token


@pytest.mark.parametrize("delta,flagged", [(5e-5, True), (-5e-5, True), (2e-4, False), (-2e-4, False)])
def test_sampler_cdf_edge_flag(delta, flagged):
    z = np.log([[0.1, 0.2, 0.3, 0.4]]).astype(np.float32)
    edge = np.cumsum(_dist(z[0], 1.0))[1]   # 0.3
    tok, flags = oracle.sample_draft(z, "f32", np.ones(1, np.float32),
                                     np.array([edge + delta], np.float32))
    assert bool(flags[0] & oracle.TIE_CDF) == flagged
    assert tok[0] == (2 if edge + delta > edge else 1)


def test_sampler_flags_unusable_rows():
    z = np.zeros((3, 4), np.float32)
    z[2] = -np.inf
    tok, flags = oracle.sample_draft(z, "f32", np.array([-1.0, 1.0, 1.0], np.float32),
                                     np.array([0.5, 1.0, 0.5], np.float32))
    assert np.all(tok == -1) and np.all(flags & oracle.BAD_INPUT)


# ---------------------------------------------------------------- one-hot draft


def _onehot_inp(zp, x, u, ur, T=1.0, dtype="f32"):
    zp = np.asarray(zp)
    B = len(x)
    K = len(x[0])
    tgt = np.ascontiguousarray(np.broadcast_to(zp, (B,) + zp.shape))
    return dict(B=B, K=K, V=zp.shape[-1], dtype=dtype, target=tgt, draft=None,
                draft_tokens=np.asarray(x, np.int32).reshape(B, K), draft_len=None,
                temperature=np.full(B, T, np.float32),
                uniforms=np.asarray(u, np.float32).reshape(B, K + 1),
                uniforms_resample=np.asarray(ur, np.float32).reshape(B))


@pytest.mark.parametrize("seed,V,K,T", [(21, 4, 2, 1.0), (22, 6, 1, 0.7), (23, 3, 3, 1.3)])
def test_onehot_exact_law_is_p(seed, V, K, T):
    """For any fixed drafts x (the draft's top tokens), the emitted law is
    p: token 0 ~ p_0, reaching t has probability prod_{s<t} p_s(x_s), and the
    token at t given reaching t ~ p_t."""
    rng = np.random.default_rng(seed)
    zp = (1.5 * rng.standard_normal((K + 1, V))).astype(np.float32)
    p = [_dist(zp[t], T) for t in range(K + 1)]
    for x in itertools.product(range(V), repeat=K):
        us, urs, ws = [], [], []
        res_mids = []
        for t in range(K):
            w = p[t].copy()
            w[x[t]] = 0.0
            res_mids.append(_mid_intervals(np.cumsum(w / w.sum())[:-1]))
        b_mid, b_len = _mid_intervals(np.cumsum(p[K])[:-1])
        for pattern in itertools.product((True, False), repeat=K):
            ut, lt = [], 1.0
            for t in range(K):
                r = p[t][x[t]]
                a, bb = (0.0, r) if pattern[t] else (r, 1.0)
                ut.append((a + bb) / 2)
                lt *= bb - a
            if lt == 0:
                continue
            j = next((t for t in range(K) if not pattern[t]), K)
            finals = list(zip(*res_mids[j])) if j < K else list(zip(b_mid, b_len))
            for m, ln in finals:
                u = np.zeros(K + 1)
                u[:K] = ut
                if j == K:
                    u[K] = m
                us.append(u)
                urs.append(m if j < K else 0.5)
                ws.append(lt * ln)
        inp = _onehot_inp(zp, [x] * len(us), us, urs, T)
        acc, out, flags = oracle.verify_onehot(inp)
        assert np.all(flags & oracle.BAD_INPUT == 0)
        law0 = np.zeros(V)
        np.add.at(law0, out[:, 0], ws)
        assert np.max(np.abs(law0 - p[0])) < 1e-6
        reach = np.cumprod([1.0] + [p[t][x[t]] for t in range(K)])
        for t in range(K + 1):
            sel = acc >= t
            assert abs(np.sum(np.asarray(ws)[sel]) - reach[t]) < 1e-6
            lawt = np.zeros(V)
            np.add.at(lawt, out[sel, t], np.asarray(ws)[sel])
            assert np.max(np.abs(lawt - reach[t] * p[t])) < 1e-6


def test_onehot_equals_general_rule_with_point_mass_draft():
    """The general rule with draft logits that are -inf except at x (so q is
    exactly the point mass) gives the same outputs as the one-hot rule."""
    rng = np.random.default_rng(31)
    B, K, V = 600, 3, 12
    inp = synth.random_case(31, B, K, V, "f32", temperature=0.9, draft_len="random")
    x = inp["draft_tokens"]
    zq = np.full((B, K, V), -np.inf, np.float32)
    for t in range(K):
        zq[np.arange(B), t, x[:, t]] = 0.0
    general = dict(inp, draft=zq)
    acc_g, out_g, fl_g = oracle.verify_sample(general)
    acc_o, out_o, fl_o = oracle.verify_onehot(inp)
    assert np.array_equal(acc_g, acc_o) and np.array_equal(out_g, out_o)
    assert np.all(fl_o & oracle.BAD_INPUT == 0)


def test_onehot_greedy_matches_greedy_rule():
    inp = synth.random_case(32, 200, 4, 30, "f32", temperature=0.0, draft_len="random")
    acc_g, out_g, _ = oracle.verify_sample(dict(inp, draft=None))
    acc_o, out_o, _ = oracle.verify_onehot(inp)
    assert np.array_equal(acc_g, acc_o) and np.array_equal(out_g, out_o)


@pytest.mark.parametrize("delta,flagged", [(5e-5, True), (-5e-5, True), (2e-4, False), (-2e-4, False)])
def test_onehot_accept_tie_flag(delta, flagged):
    zp = np.log([[0.25, 0.5, 0.25], [1 / 3, 1 / 3, 1 / 3]]).astype(np.float32)
    px = _dist(zp[0], 1.0)[1]
    inp = _onehot_inp(zp, [[1]], [[px + delta, 0.1]], [0.2])
    acc, out, flags = oracle.verify_onehot(inp)
    assert bool(flags[0] & oracle.TIE_ACCEPT) == flagged
    assert acc[0] == (1 if px + delta < px else 0)
    if acc[0] == 0:
        assert out[0, 0] != 1      # the rejected token is never the replacement


# ---------------------------------------------------------------- greedy token tree


def _brute_tree(z, parents, tokens, n):
    """Every root-to-node path checked edge by edge with numpy's argmax; the
    deepest fully-agreeing node (lowest index among the deepest)."""
    g = np.argmax(z[:n], axis=1)
    best, best_depth = 0, 0
    for v in range(1, n):
        path, u = [], v
        while u != 0:
            path.append(u)
            u = parents[u]
        ok = all(tokens[w] == g[parents[w]] for w in path)
        if ok and len(path) > best_depth:
            best, best_depth = v, len(path)
    nodes = []
    u = best
    while u != 0:
        nodes.append(u)
        u = parents[u]
    nodes = nodes[::-1]
    return best_depth, [tokens[w] for w in nodes] + [g[best]], [0] + nodes


def _random_tree(rng, N, V, agree=0.6):
    parents = np.full(N, -1, np.int32)
    for i in range(1, N):
        parents[i] = rng.integers(0, i)
    z = rng.integers(-2, 3, size=(N, V)).astype(np.float32)
    g = np.argmax(z, axis=1)
    tokens = np.zeros(N, np.int32)
    for i in range(1, N):
        tokens[i] = g[parents[i]] if rng.random() < agree else rng.integers(0, V)
    return z, parents, tokens


def test_tree_brute_force_small_trees():
    rng = np.random.default_rng(41)
    B, N, V = 300, 9, 6
    zs, ps, ts, ns = [], [], [], []
    for b in range(B):
        z, par, tok = _random_tree(rng, N, V)
        zs.append(z)
        ps.append(par)
        ts.append(tok)
        ns.append(rng.integers(1, N + 1))
    acc, out, path = oracle.tree_greedy(np.stack(zs), "f32", np.stack(ps), np.stack(ts), np.array(ns))
    for b in range(B):
        d, toks, nodes = _brute_tree(zs[b], ps[b], ts[b], ns[b])
        assert acc[b] == d
        assert list(out[b, :d + 1]) == toks and np.all(out[b, d + 1:] == -1)
        assert list(path[b, :d + 1]) == nodes and np.all(path[b, d + 1:] == -1)


def test_tree_chain_equals_linear_greedy_rule():
    """A chain tree (parent of node i is i - 1) is the linear step: the same
    outputs as the greedy verification rule with drafts tokens[1..n-1]."""
    inp = synth.random_case(42, 300, 5, 20, "f32", temperature=0.0, draft_len="random")
    B, K, V = inp["B"], inp["K"], inp["V"]
    z = synth.bf16_to_f32(synth.bf16_bits(np.round(inp["target"] * 2) / 2))
    inp["target"] = z
    acc_l, out_l, _ = oracle.verify_sample(dict(inp, draft=None))
    parents = np.tile(np.arange(-1, K, dtype=np.int32), (B, 1))
    tokens = np.concatenate([np.zeros((B, 1), np.int32), inp["draft_tokens"]], axis=1)
    acc_t, out_t, path_t = oracle.tree_greedy(z, "f32", parents, tokens, inp["draft_len"] + 1)
    assert np.array_equal(acc_t, acc_l)
    assert np.array_equal(out_t, out_l)
    for b in range(B):
        assert list(path_t[b, :acc_t[b] + 1]) == list(range(acc_t[b] + 1))


def test_tree_star_picks_lowest_matching_child():
    V = 5
    z = np.zeros((1, 4, V), np.float32)
    z[0, 0, 3] = 1.0                       # argmax at the root: token 3
    z[0, 2, 1] = 1.0
    z[0, 3, 4] = 1.0
    parents = np.array([[-1, 0, 0, 0]], np.int32)
    tokens = np.array([[0, 2, 3, 3]], np.int32)   # nodes 2 and 3 both agree
    acc, out, path = oracle.tree_greedy(z, "f32", parents, tokens, np.array([4]))
    assert acc[0] == 1 and list(out[0]) == [3, 1, -1, -1] and list(path[0]) == [0, 2, -1, -1]


def test_tree_rejects_malformed_trees():
    z = np.zeros((3, 3, 4), np.float32)
    parents = np.array([[-1, 0, 1], [-1, 1, 0], [0, 0, 1]], np.int32)
    tokens = np.zeros((3, 3), np.int32)
    acc, out, path = oracle.tree_greedy(z, "f32", parents, tokens, np.array([3, 3, 3]))
    assert acc[0] == 2 and list(acc[1:]) == [-1, -1]
    acc, _, _ = oracle.tree_greedy(z, "f32", parents, tokens, np.array([0, 4, 1]))
    assert list(acc) == [-1, -1, -1]


# ---------------------------------------------------------------- post-accept insert


def _golden():
    rows = {}
    with open(os.path.join(GOLDEN, "post_accept_insert.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, *v = line.split()
                rows[k] = np.array([int(x) for x in v], np.int32)
    return rows


def test_insert_worked_example():
    g = _golden()
    B = len(g["accepted_len"])
    out = np.stack([g[f"out_tokens_{b}"] for b in range(B)])
    hist = np.stack([g[f"history_{b}"] for b in range(B)])
    seq, hist2, nxt, cu, packed, status = oracle.insert_accepted(g["accepted_len"], out,
                                                                 g["seq_lens"], hist)
    assert np.array_equal(seq, g["exp_seq_lens"])
    assert np.array_equal(hist2, np.stack([g[f"exp_history_{b}"] for b in range(B)]))
    assert np.array_equal(nxt, g["exp_next_tokens"])
    assert np.array_equal(cu, g["exp_cu_emitted"])
    assert np.array_equal(packed[:cu[-1]], g["exp_packed"])
    assert np.array_equal(status, g["exp_status"])


def test_insert_invariants_random():
    rng = np.random.default_rng(51)
    B, K, L = 500, 6, 40
    acc = rng.integers(-1, K + 1, size=B).astype(np.int32)
    out = rng.integers(0, 1000, size=(B, K + 1)).astype(np.int32)
    seq = rng.integers(0, L, size=B).astype(np.int32)
    hist = rng.integers(0, 1000, size=(B, L)).astype(np.int32)
    seq2, hist2, nxt, cu, packed, status = oracle.insert_accepted(acc, out, seq, hist)
    emitted = np.where(status == 0, acc + 1, 0)
    assert np.array_equal(np.diff(cu), emitted) and cu[0] == 0
    assert np.array_equal(seq2, seq + emitted)
    for b in range(B):
        assert np.array_equal(hist2[b, :seq[b]], hist[b, :seq[b]])          # history kept
        assert np.array_equal(hist2[b, seq2[b]:], hist[b, seq2[b]:])        # nothing past it
        if status[b] == 0:
            assert np.array_equal(hist2[b, seq[b]:seq2[b]], out[b, :acc[b] + 1])
            assert np.array_equal(packed[cu[b]:cu[b + 1]], out[b, :acc[b] + 1])
            assert nxt[b] == out[b, acc[b]]
        else:
            assert nxt[b] == -1
            assert status[b] == (1 if not 0 <= acc[b] <= K else 2)
