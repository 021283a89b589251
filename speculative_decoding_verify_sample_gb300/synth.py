"""Seeded synthetic inputs for the verification sampler.

This module builds inputs only: logits, drafted tokens, draft lengths,
temperatures and the uniforms the sampler consumes.  It holds none of the
sampler's arithmetic (no normaliser, no accept test, no inverse CDF, no target
argmax), so the CUDA path and the CPU oracle can both be fed from it without
sharing any of the method.

* Normals and uniforms come from numpy's PCG64 generator, seeded per workload;
  the uniforms the sampler consumes come from an independent stream
  (seed + 1000) and are multiples of 2^-24 in [0, 1), exact in fp32 and fp64.
* Drafted tokens x ~ softmax(z_q / T) are drawn with the Gumbel-max trick
  (argmax of z_q/T + Gumbel noise), a draw from the draft distribution that
  needs no normaliser.  A T = 0 request drafts the draft row's own argmax.
* bf16 logits are rounded from fp32 with round-to-nearest-even and stored as
  raw uint16.
* The greedy workload draws target logits N(0, 3^2) in bf16 with nothing
  planted, so exact ties at a row's maximum occur (about one row in ten at
  V = 128256).  The draft model is the target itself at a position with
  probability 0.8 and an independent N(0, 3^2) row otherwise, and it
  proposes its own top token (lowest index on ties), so the drafted token
  is the target's argmax with probability about 0.8.
* The planted greedy workload instead gives every target row the value 16.0
  at a random index g and clips every other entry to at most 15.9375, so
  argmax = g by construction; the draft token is g with probability 0.8 and
  otherwise uniform over the other V - 1 tokens.
* The long ragged workload uses constant-overlap pairs: r = softmax(3 * N(0,1))
  over V, a random half A of the vocabulary and its complement A', and
  p = alpha*r + (1-alpha)*r|A, q = alpha*r + (1-alpha)*r|A' (each restriction
  renormalised).  Then min(p, q) = alpha*r pointwise, so sum min(p, q) = alpha
  exactly, and the logits are log p, log q in fp32.

Workload shapes follow the pages' model families (Llama-3-class V = 128256,
DeepSeek-class V = 129280, draft lengths 1..8).
"""

from __future__ import annotations

import numpy as np

WORKLOADS = {
    # name: (B, K, V, dtype)
    "tiny": (4, 4, 1024, "f32"),
    "tiny_greedy": (4, 4, 1024, "f32"),
    "llama3": (32, 4, 128256, "bf16"),
    "greedy": (256, 4, 128256, "bf16"),
    "greedy_planted": (256, 4, 128256, "bf16"),
    "dsv3_mtp": (512, 1, 129280, "bf16"),
    "ragged": (128, 8, 128256, "f32"),
}

DEFAULT_SEED = {"tiny": 0, "tiny_greedy": 0, "llama3": 1, "greedy": 2, "dsv3_mtp": 3, "ragged": 4,
                "greedy_planted": 5}

RAGGED_ALPHAS = (0.5, 0.8, 0.95)

_ROW_CHUNK = 64


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 (round to nearest even), as raw uint16 bits. Finite inputs."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    u = u + (((u >> 16) & 1) + np.uint32(0x7FFF))
    return (u >> 16).astype(np.uint16)


def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    """Raw bf16 bits -> float32 (exact)."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def as_f32(logits: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_to_f32(logits) if dtype == "bf16" else np.asarray(logits, np.float32)


def uniforms24(rng: np.random.Generator, shape) -> np.ndarray:
    """Uniforms on the 2^-24 grid in [0, 1): exact in fp32."""
    return (rng.integers(0, 1 << 24, size=shape, dtype=np.int64).astype(np.float64)
            * 2.0 ** -24).astype(np.float32)


def gumbel_draw(rng: np.random.Generator, z: np.ndarray, T: np.ndarray) -> np.ndarray:
    """One token per row of z [R, V] from softmax(z / T[r]) by Gumbel-max;
    rows with T == 0 take their own argmax.  Returns int32 [R]."""
    R = z.shape[0]
    out = np.empty(R, np.int32)
    for lo in range(0, R, _ROW_CHUNK):
        hi = min(R, lo + _ROW_CHUNK)
        tt = np.asarray(T[lo:hi], np.float64)
        if not np.any(tt > 0):     # every row drafts its own top token: no noise drawn
            out[lo:hi] = np.argmax(np.asarray(z[lo:hi]), axis=1)
            continue
        zz = np.asarray(z[lo:hi], np.float64)
        u = rng.random(zz.shape)
        g = -np.log(-np.log(np.clip(u, 1e-300, 1.0 - 1e-16)))
        hot = tt > 0
        scaled = np.where(hot[:, None], zz / np.where(hot, tt, 1.0)[:, None] + g, zz)
        out[lo:hi] = np.argmax(scaled, axis=1)
    return out


def _pack(B, K, V, dtype, target, draft, tokens, draft_len, temperature, urng, **extra):
    inp = dict(B=B, K=K, V=V, dtype=dtype, target=target, draft=draft,
               draft_tokens=np.ascontiguousarray(tokens, np.int32).reshape(B, K),
               draft_len=None if draft_len is None else np.ascontiguousarray(draft_len, np.int32),
               temperature=np.ascontiguousarray(temperature, np.float32),
               uniforms=uniforms24(urng, (B, K + 1)),
               uniforms_resample=uniforms24(urng, (B,)))
    inp.update(extra)
    return inp


def _noisy_pair(rng, rows_t, rows_d, V, scale, noise, dtype):
    """Draft logits ~ N(0, scale^2); target = draft + N(0, noise^2).  The target
    has K+1 rows per request, the draft K; the extra target row gets its own
    draft-like base."""
    B, K1 = rows_t
    K = rows_d[1]
    zq_all = (scale * rng.standard_normal((B, K1, V), dtype=np.float32))
    zp = zq_all + np.float32(noise) * rng.standard_normal((B, K1, V), dtype=np.float32)
    zq = zq_all[:, :K, :]
    if dtype == "bf16":
        return bf16_bits(zp), bf16_bits(zq)
    return np.ascontiguousarray(zp), np.ascontiguousarray(zq)


def _tiny(seed, greedy):
    B, K, V, dt = WORKLOADS["tiny"]
    rng = np.random.default_rng(seed)
    urng = np.random.default_rng(seed + 1000)
    tgt, drf = _noisy_pair(rng, (B, K + 1), (B, K), V, 2.0, 0.5, dt)
    T = np.ones(B, np.float32)
    toks = gumbel_draw(rng, drf.reshape(B * K, V), np.repeat(T, K))
    if greedy:
        T = np.zeros(B, np.float32)
    return _pack(B, K, V, dt, tgt, drf, toks, None, T, urng)


def _llama3(seed):
    B, K, V, dt = WORKLOADS["llama3"]
    rng = np.random.default_rng(seed)
    urng = np.random.default_rng(seed + 1000)
    tgt, drf = _noisy_pair(rng, (B, K + 1), (B, K), V, 3.0, 1.0, dt)
    T = np.full(B, 0.7, np.float32)
    toks = gumbel_draw(rng, bf16_to_f32(drf).reshape(B * K, V), np.repeat(T, K))
    return _pack(B, K, V, dt, tgt, drf, toks, None, T, urng)


def _greedy(seed):
    B, K, V, dt = WORKLOADS["greedy"]
    rng = np.random.default_rng(seed)
    urng = np.random.default_rng(seed + 1000)
    tgt = bf16_bits(3.0 * rng.standard_normal((B, K + 1, V), dtype=np.float32))
    # the draft model: the target's own row at a position w.p. 0.8, else an
    # independent row; it proposes its top token (T = 0 drafting)
    same = rng.random((B, K)) < 0.8
    toks = np.empty((B, K), np.int32)
    for b in range(B):
        rows = bf16_to_f32(tgt[b, :K]).copy()
        other = ~same[b]
        if other.any():
            rows[other] = bf16_to_f32(bf16_bits(
                3.0 * rng.standard_normal((int(other.sum()), V), dtype=np.float32)))
        toks[b] = gumbel_draw(rng, rows, np.zeros(K))
    T = np.zeros(B, np.float32)
    return _pack(B, K, V, dt, tgt, None, toks, None, T, urng, draft_is_target=same)


def _greedy_planted(seed):
    B, K, V, dt = WORKLOADS["greedy_planted"]
    rng = np.random.default_rng(seed)
    urng = np.random.default_rng(seed + 1000)
    z = 3.0 * rng.standard_normal((B, K + 1, V), dtype=np.float32)
    np.clip(z, -16.0, 15.9375, out=z)
    g = rng.integers(0, V, size=(B, K + 1))
    bi, ti = np.meshgrid(np.arange(B), np.arange(K + 1), indexing="ij")
    z[bi, ti, g] = 16.0
    tgt = bf16_bits(z)
    del z
    hit = rng.random((B, K)) < 0.8
    other = rng.integers(0, V - 1, size=(B, K))
    other = other + (other >= g[:, :K])
    toks = np.where(hit, g[:, :K], other).astype(np.int32)
    T = np.zeros(B, np.float32)
    return _pack(B, K, V, dt, tgt, None, toks, None, T, urng, planted_argmax=g.astype(np.int32))


def _dsv3(seed):
    B, K, V, dt = WORKLOADS["dsv3_mtp"]
    rng = np.random.default_rng(seed)
    urng = np.random.default_rng(seed + 1000)
    tgt, drf = _noisy_pair(rng, (B, K + 1), (B, K), V, 3.0, 0.7, dt)
    T = (1.2 * (1.0 - uniforms24(rng, (B,)).astype(np.float64))).astype(np.float32)
    T[rng.permutation(B)[: B // 4]] = 0.0
    toks = gumbel_draw(rng, bf16_to_f32(drf).reshape(B * K, V), np.repeat(T, K))
    return _pack(B, K, V, dt, tgt, drf, toks, None, T, urng)


def constant_overlap_rows(rng, rows: int, V: int, alpha: np.ndarray, sigma: float = 3.0):
    """log p, log q (float32 [rows, V]) with sum_i min(p_i, q_i) = alpha[r]."""
    logp = np.empty((rows, V), np.float32)
    logq = np.empty((rows, V), np.float32)
    for lo in range(0, rows, _ROW_CHUNK):
        hi = min(rows, lo + _ROW_CHUNK)
        n = hi - lo
        s = sigma * rng.standard_normal((n, V))
        s -= s.max(axis=1, keepdims=True)
        r = np.exp(s)
        r /= r.sum(axis=1, keepdims=True)
        inA = np.zeros((n, V), bool)
        perm = np.argsort(rng.random((n, V)), axis=1)[:, : V // 2]
        np.put_along_axis(inA, perm, True, axis=1)
        rA = np.where(inA, r, 0.0)
        rA /= rA.sum(axis=1, keepdims=True)
        rB = np.where(inA, 0.0, r)
        rB /= rB.sum(axis=1, keepdims=True)
        a = np.asarray(alpha[lo:hi], np.float64)[:, None]
        logp[lo:hi] = np.log(a * r + (1.0 - a) * rA)
        logq[lo:hi] = np.log(a * r + (1.0 - a) * rB)
    return logp, logq


def _ragged(seed):
    B, K, V, dt = WORKLOADS["ragged"]
    rng = np.random.default_rng(seed)
    urng = np.random.default_rng(seed + 1000)
    alpha_b = np.array([RAGGED_ALPHAS[b % len(RAGGED_ALPHAS)] for b in range(B)])
    n = rng.integers(1, K + 1, size=B).astype(np.int32)
    logp, logq = constant_overlap_rows(rng, B * (K + 1), V, np.repeat(alpha_b, K + 1))
    tgt = logp.reshape(B, K + 1, V)
    drf = np.ascontiguousarray(logq.reshape(B, K + 1, V)[:, :K, :])
    del logq
    T = np.ones(B, np.float32)
    toks = gumbel_draw(rng, drf.reshape(B * K, V), np.repeat(T, K))
    return _pack(B, K, V, dt, tgt, drf, toks, n, T, urng, alpha=alpha_b)


def make_inputs(name: str, seed: int | None = None) -> dict:
    """Inputs for one named workload, as host numpy arrays (see module doc)."""
    if seed is None:
        seed = DEFAULT_SEED[name]
    if name in ("tiny", "tiny_greedy"):
        return _tiny(seed, name == "tiny_greedy")
    return {"llama3": _llama3, "greedy": _greedy, "greedy_planted": _greedy_planted,
            "dsv3_mtp": _dsv3, "ragged": _ragged}[name](seed)


def random_case(seed: int, B: int, K: int, V: int, dtype: str = "f32", *, scale: float = 2.0,
                noise: float = 0.5, temperature=1.0, draft_len=None, greedy_frac: float = 0.0,
                draft_greedy_frac: float = 0.0) -> dict:
    """A small random case of any shape: draft ~ N(0, scale^2), target = draft +
    N(0, noise^2), drafted tokens ~ q (Gumbel-max).  ``temperature`` is a
    scalar or per-request array; ``greedy_frac`` of the requests get T = 0;
    ``draft_len`` None (all K), "random" (uniform 1..K) or an array."""
    rng = np.random.default_rng(seed)
    urng = np.random.default_rng(seed + 1000)
    tgt, drf = _noisy_pair(rng, (B, K + 1), (B, K), V, scale, noise, dtype)
    T = np.broadcast_to(np.asarray(temperature, np.float32), (B,)).copy()
    if greedy_frac > 0:
        T[rng.random(B) < greedy_frac] = 0.0
    dl = None
    if isinstance(draft_len, str) and draft_len == "random":
        dl = rng.integers(1, K + 1, size=B).astype(np.int32)
    elif draft_len is not None:
        dl = np.broadcast_to(np.asarray(draft_len, np.int32), (B,)).copy()
    zq = as_f32(drf, dtype).reshape(B * K, V)
    Tdraw = np.repeat(T, K).astype(np.float64)
    if draft_greedy_frac > 0:
        Tdraw[rng.random(B * K) < draft_greedy_frac] = 0.0
    toks = gumbel_draw(rng, zq, np.where(Tdraw > 0, np.maximum(Tdraw, 1e-3), 0.0))
    return _pack(B, K, V, dtype, tgt, drf, toks, dl, T, urng)


def rows_needed(inp: dict):
    """(target rows, draft rows) the rule must stream for these inputs:
    target rows t <= n_b for every request, draft rows t < n_b for T_b > 0
    when draft logits are given (the one-hot rule has none)."""
    B, K = inp["B"], inp["K"]
    n = np.full(B, K) if inp.get("draft_len") is None else np.asarray(inp["draft_len"])
    T = np.asarray(inp["temperature"])
    rows_d = int(np.sum(np.where(T > 0, n, 0))) if inp.get("draft") is not None else 0
    return int(np.sum(n + 1)), rows_d


def draft_rows(seed: int, R: int, V: int, dtype: str = "bf16", *, scale: float = 3.0,
               greedy_frac: float = 0.25, t_max: float = 1.2) -> dict:
    """Inputs of the draft-side sampler: R rows of draft logits N(0, scale^2),
    per-row T uniform in (0, t_max] with greedy_frac of the rows at T = 0,
    and one uniform per row (the DeepSeek-class MTP draft step at
    R = 512, V = 129280)."""
    rng = np.random.default_rng(seed)
    urng = np.random.default_rng(seed + 1000)
    z = (scale * rng.standard_normal((R, V), dtype=np.float32))
    logits = bf16_bits(z) if dtype == "bf16" else np.ascontiguousarray(z)
    T = (t_max * (1.0 - uniforms24(rng, (R,)).astype(np.float64))).astype(np.float32)
    T[rng.permutation(R)[: int(round(greedy_frac * R))]] = 0.0
    return dict(R=R, V=V, dtype=dtype, logits=logits, temperature=T,
                uniforms=uniforms24(urng, (R,)))


def onehot_case(seed: int, B: int, K: int, V: int, dtype: str = "bf16", *, temperature=0.7,
                draft_len=None, greedy_frac: float = 0.0) -> dict:
    """Inputs of the one-hot (top-token) draft rule: target = draft + noise
    as in random_case, and each drafted token is the draft row's own top
    token (the draft logits are then dropped: the rule takes none)."""
    inp = random_case(seed, B, K, V, dtype, scale=3.0, noise=1.0, temperature=temperature,
                      draft_len=draft_len, greedy_frac=greedy_frac, draft_greedy_frac=1.0)
    inp["draft"] = None
    return inp


def tree_case(seed: int, B: int, N: int, V: int, dtype: str = "bf16", *, agree: float = 0.7,
              n_nodes=None, scale: float = 3.0) -> dict:
    """Token trees for greedy tree verification: node i >= 1 gets a parent
    uniform in [0, i) (random recursive trees), target logits N(0, scale^2)
    per node.  A node's token is drafted by a draft model that, with
    probability `agree`, scores its parent position exactly as the target
    does and proposes its top token (lowest index); otherwise it proposes a
    uniform token.  n_nodes: None (all N) or "random" (uniform 1..N)."""
    rng = np.random.default_rng(seed)
    z = scale * rng.standard_normal((B, N, V), dtype=np.float32)
    logits = bf16_bits(z) if dtype == "bf16" else np.ascontiguousarray(z)
    del z
    parents = np.full((B, N), -1, np.int32)
    for i in range(1, N):
        parents[:, i] = rng.integers(0, i, size=B)
    tokens = rng.integers(0, V, size=(B, N)).astype(np.int32)
    tokens[:, 0] = 0
    same = rng.random((B, N)) < agree
    same[:, 0] = False
    for b in range(B):
        idx = np.nonzero(same[b])[0]
        if len(idx):
            rows = as_f32(logits[b, parents[b, idx]], dtype)   # the draft's copy of the parent rows
            tokens[b, idx] = gumbel_draw(rng, rows, np.zeros(len(idx)))
    if n_nodes is None:
        nn = np.full(B, N, np.int32)
    elif isinstance(n_nodes, str) and n_nodes == "random":
        nn = rng.integers(1, N + 1, size=B).astype(np.int32)
    else:
        nn = np.broadcast_to(np.asarray(n_nodes, np.int32), (B,)).copy()
    return dict(B=B, N=N, V=V, dtype=dtype, target=logits, parents=parents, tokens=tokens,
                n_nodes=nn)
