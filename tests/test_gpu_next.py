"""The CUDA path of the steps around verification against the oracle,
through the C ABI: the draft-side sampler, the one-hot (top-token) draft
rule, greedy token-tree verification and the post-accept insert.

Rules as for the verification step (tests/helpers.py): greedy bit-exact,
sampled draws equal except at oracle-flagged near-ties (counted, capped),
per-row maxima exact and normalisers within 1e-5 relative; the tree and the
insert are integer results, bit-exact.
"""

import numpy as np
import pytest

import oracle
from helpers import PROB_RTOL, assert_outputs_match, excuse_ceiling, report_parity
from speculative_decoding_verify_sample_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verify_sample_gb300 as sv
    sv.build()
    sv.lib()


def _logits(a, dtype):
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()


def _i32(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()


def _f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()


# ---------------------------------------------------------------- draft-side sampler


def _check_sampler(d, label, stats_rows=None):
    import speculative_decoding_verify_sample_gb300 as sv
    R, V = d["R"], d["V"]
    rs = torch.full((R, 8), float("nan"), device="cuda")
    tok = sv.sample_draft(_logits(d["logits"], d["dtype"]), _f32(d["temperature"]),
                          _f32(d["uniforms"]), row_stats=rs)
    torch.cuda.synchronize()
    tok = tok.cpu().numpy()
    rs = rs.cpu().numpy().astype(np.float64)
    tok_o, flags_o = oracle.sample_draft(d["logits"], d["dtype"], d["temperature"], d["uniforms"],
                                         nthreads=16)
    T = d["temperature"]
    mism = tok != tok_o
    assert not np.any(mism & (T == 0)), np.nonzero(mism & (T == 0))[0][:8]
    allowed = (flags_o & oracle.NEAR_TIE_MASK) != 0
    assert not np.any(mism & ~allowed), np.nonzero(mism & ~allowed)[0][:8]
    excused = int((mism & allowed).sum())
    report_parity({"label": label, "compared": R, "sampled": int((T > 0).sum()),
                   "excused": excused,
                   "flagged": {name: int(((flags_o & bit) != 0).sum())
                               for bit, name in oracle.FLAG_NAMES.items()}})
    assert excused <= excuse_ceiling(int((T > 0).sum()))
    # per-row maxima and normalisers (a row of the sampler is the verify's bonus row)
    z = synth.as_f32(d["logits"], d["dtype"]).astype(np.float64)
    rows = np.arange(R) if stats_rows is None else stats_rows
    for r in rows:
        assert rs[r, 0] == z[r].max(), (r, rs[r, 0], z[r].max())
        if T[r] > 0:
            Tr = float(np.float32(T[r]))
            S = np.exp((z[r] - z[r].max()) / Tr).sum()
            assert abs(rs[r, 1] - S) <= PROB_RTOL * S, (r, rs[r, 1], S)
        assert rs[r, 7] == tok[r]


@pytest.mark.parametrize("seed,R,V,dtype", [(1, 37, 1000, "f32"), (2, 64, 50257, "bf16"),
                                            (3, 9, 70001, "bf16"), (4, 20, 3, "f32"),
                                            (5, 33, 200001, "f32")])
def test_sampler_random(seed, R, V, dtype):
    _check_sampler(synth.draft_rows(seed, R, V, dtype, greedy_frac=0.3), f"sampler{seed}")


def test_sampler_full_dsv3_draft_step():
    d = synth.draft_rows(6, 512, 129280, "bf16")
    _check_sampler(d, "sampler_dsv3", stats_rows=np.arange(0, 512, 4))


def test_sampler_flags_bad_rows():
    import speculative_decoding_verify_sample_gb300 as sv
    d = synth.draft_rows(7, 6, 500, "f32", greedy_frac=0.0)
    d["temperature"][1] = -1.0
    d["uniforms"][2] = 1.0
    d["logits"][3] = -np.inf
    ws = sv.Workspace(6, 0, 500, "f32", "cuda", kind="sample")
    tok = sv.sample_draft(_logits(d["logits"], "f32"), _f32(d["temperature"]),
                          _f32(d["uniforms"]), workspace=ws)
    torch.cuda.synchronize()
    tok = tok.cpu().numpy()
    assert list(tok[1:4]) == [-1, -1, -1]
    st = ws.read_status()
    assert st & sv.DEV_BAD_TEMPERATURE and st & sv.DEV_BAD_UNIFORM and st & sv.DEV_BAD_ROW
    tok_o, _ = oracle.sample_draft(d["logits"], "f32", d["temperature"], d["uniforms"])
    assert list(tok_o[1:4]) == [-1, -1, -1]
    good = [0, 4, 5]
    assert np.array_equal(tok[good], tok_o[good])


# ---------------------------------------------------------------- one-hot draft


def _run_onehot(inp, ws=None, debug=False):
    import speculative_decoding_verify_sample_gb300 as sv
    B, K = inp["B"], inp["K"]
    rs = torch.full((B, K + 1, 8), float("nan"), device="cuda") if debug else None
    acc, out = sv.spec_verify_sample_onehot(
        _logits(inp["target"], inp["dtype"]), _i32(inp["draft_tokens"]), _i32(inp.get("draft_len")),
        _f32(inp["temperature"]), _f32(inp["uniforms"]), _f32(inp["uniforms_resample"]),
        workspace=ws, row_stats=rs)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), out.cpu().numpy(), (rs.cpu().numpy() if debug else None)


@pytest.mark.parametrize("seed,B,K,V,dtype,T,dl,gf", [
    (11, 16, 4, 1000, "f32", 1.0, None, 0.0),
    (12, 24, 6, 50257, "bf16", 0.8, "random", 0.3),
    (13, 7, 3, 70001, "bf16", 1.2, "random", 0.0),
    (14, 5, 16, 3001, "f32", 0.5, "random", 0.2),
    (15, 9, 2, 8, "f32", 1.0, None, 0.0),
])
def test_onehot_random(seed, B, K, V, dtype, T, dl, gf):
    inp = synth.onehot_case(seed, B, K, V, dtype, temperature=T, draft_len=dl, greedy_frac=gf)
    acc_o, out_o, flags_o = oracle.verify_onehot(inp, nthreads=8)
    acc, out, rs = _run_onehot(inp, debug=True)
    assert_outputs_match(inp, acc, out, acc_o, out_o, flags_o, label=f"onehot{seed}")
    # a rejected drafted token is never its own replacement
    for b in range(B):
        n = K if inp["draft_len"] is None else inp["draft_len"][b]
        if 0 <= acc[b] < n and inp["temperature"][b] > 0:
            assert out[b, acc[b]] != inp["draft_tokens"][b, acc[b]]


def test_onehot_full_batch():
    inp = synth.onehot_case(16, 128, 4, 128256, "bf16", temperature=0.7, greedy_frac=0.25)
    acc_o, out_o, flags_o = oracle.verify_onehot(inp, nthreads=16)
    acc, out, _ = _run_onehot(inp)
    assert_outputs_match(inp, acc, out, acc_o, out_o, flags_o, label="onehot_full")


def test_onehot_dominant_token_rejection():
    # p(x) = 0.9 at the drafted token: a rejection draws from the other 10 %
    V, B = 64, 40
    rng = np.random.default_rng(17)
    z = rng.standard_normal((B, 2, V)).astype(np.float32)
    z[:, 0, 5] = np.log(0.9) - np.log(0.1) + np.log(np.exp(z[:, 0, :]).sum(1) - np.exp(z[:, 0, 5]))
    u = synth.uniforms24(rng, (B, 2))
    u[:, 0] = 0.9 + 0.1 * u[:, 0]          # mostly above p(x): rejected
    inp = dict(B=B, K=1, V=V, dtype="f32", target=z, draft=None,
               draft_tokens=np.full((B, 1), 5, np.int32), draft_len=None,
               temperature=np.ones(B, np.float32), uniforms=u.astype(np.float32),
               uniforms_resample=synth.uniforms24(rng, (B,)))
    acc_o, out_o, flags_o = oracle.verify_onehot(inp)
    acc, out, _ = _run_onehot(inp)
    assert (acc_o == 0).sum() > 10
    assert_outputs_match(inp, acc, out, acc_o, out_o, flags_o, label="onehot_dominant")
    assert np.all(out[acc == 0, 0] != 5)


# ---------------------------------------------------------------- greedy token tree


def _run_tree(c, debug=False):
    import speculative_decoding_verify_sample_gb300 as sv
    B, N = c["B"], c["N"]
    rs = torch.full((B, N, 8), float("nan"), device="cuda") if debug else None
    acc, out, path = sv.verify_tree_greedy(_logits(c["target"], c["dtype"]), _i32(c["parents"]),
                                           _i32(c["tokens"]), _i32(c["n_nodes"]), row_stats=rs)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), out.cpu().numpy(), path.cpu().numpy(), rs


@pytest.mark.parametrize("seed,B,N,V,dtype,nn", [(21, 40, 12, 600, "f32", "random"),
                                                  (22, 16, 33, 50257, "bf16", None),
                                                  (23, 8, 64, 3001, "bf16", "random"),
                                                  (24, 30, 1, 100, "f32", None),
                                                  (25, 12, 20, 70001, "bf16", "random")])
def test_tree_random(seed, B, N, V, dtype, nn):
    c = synth.tree_case(seed, B, N, V, dtype, n_nodes=nn)
    acc_o, out_o, path_o = oracle.tree_greedy(c["target"], dtype, c["parents"], c["tokens"],
                                              c["n_nodes"], nthreads=8)
    acc, out, path, _ = _run_tree(c)
    assert np.array_equal(acc, acc_o) and np.array_equal(out, out_o) and np.array_equal(path, path_o)


def test_tree_ties_lowest_index():
    rng = np.random.default_rng(26)
    B, N, V = 60, 10, 9
    z = rng.integers(-2, 3, size=(B, N, V)).astype(np.float32)   # many ties at the max
    c = dict(B=B, N=N, V=V, dtype="bf16", target=synth.bf16_bits(z),
             parents=np.tile(np.r_[-1, np.arange(N - 1)], (B, 1)).astype(np.int32),
             tokens=np.zeros((B, N), np.int32), n_nodes=np.full(B, N, np.int32))
    g = np.argmax(z, axis=2)
    for b in range(B):                  # chains that follow the lowest argmax, with slips
        for i in range(1, N):
            c["tokens"][b, i] = g[b, i - 1] if rng.random() < 0.8 else rng.integers(0, V)
    acc_o, out_o, path_o = oracle.tree_greedy(c["target"], "bf16", c["parents"], c["tokens"],
                                              c["n_nodes"])
    acc, out, path, _ = _run_tree(c)
    assert np.array_equal(acc, acc_o) and np.array_equal(out, out_o) and np.array_equal(path, path_o)


def test_tree_full_size():
    c = synth.tree_case(27, 32, 32, 128256, "bf16")
    acc_o, out_o, path_o = oracle.tree_greedy(c["target"], "bf16", c["parents"], c["tokens"],
                                              c["n_nodes"], nthreads=16)
    acc, out, path, _ = _run_tree(c)
    assert np.array_equal(acc, acc_o) and np.array_equal(out, out_o) and np.array_equal(path, path_o)
    report_parity({"label": "tree_full", "compared": 32, "sampled": 0, "excused": 0,
                   "mean_accepted": float(acc.mean())})


def test_tree_malformed_flagged():
    import speculative_decoding_verify_sample_gb300 as sv
    c = synth.tree_case(28, 4, 6, 300, "f32")
    c["parents"][1, 3] = 3            # a node its own parent
    c["tokens"][2, 4] = 300           # a token outside the vocabulary
    c["n_nodes"][3] = 7               # more nodes than N
    ws = sv.Workspace(4, 6, 300, "f32", "cuda", kind="tree")
    acc, out, path = sv.verify_tree_greedy(_logits(c["target"], "f32"), _i32(c["parents"]),
                                           _i32(c["tokens"]), _i32(c["n_nodes"]), workspace=ws)
    torch.cuda.synchronize()
    acc = acc.cpu().numpy()
    assert list(acc[1:]) == [-1, -1, -1]
    st = ws.read_status()
    assert st & sv.DEV_BAD_TREE and st & sv.DEV_BAD_DRAFT_LEN
    acc_o, out_o, _ = oracle.tree_greedy(c["target"], "f32", c["parents"], c["tokens"],
                                         c["n_nodes"])
    assert acc[0] == acc_o[0] and np.array_equal(out.cpu().numpy()[0], out_o[0])


# ---------------------------------------------------------------- post-accept insert


def _insert_case(seed, B, K, L):
    rng = np.random.default_rng(seed)
    acc = rng.integers(-1, K + 2, size=B).astype(np.int32)     # some out of range
    out = rng.integers(0, 50000, size=(B, K + 1)).astype(np.int32)
    seq = rng.integers(0, L, size=B).astype(np.int32)
    hist = rng.integers(0, 50000, size=(B, L)).astype(np.int32)
    return acc, out, seq, hist


@pytest.mark.parametrize("seed,B,K,L", [(31, 7, 4, 12), (32, 3000, 8, 40), (33, 1024, 1, 4)])
def test_insert_bit_exact(seed, B, K, L):
    import speculative_decoding_verify_sample_gb300 as sv
    acc, out, seq, hist = _insert_case(seed, B, K, L)
    seq_o, hist_o, nxt_o, cu_o, packed_o, st_o = oracle.insert_accepted(acc, out, seq, hist)
    seq_d, hist_d = _i32(seq), _i32(hist)
    nxt, cu, packed, st = sv.insert_accepted(_i32(acc), _i32(out), seq_d, hist_d)
    torch.cuda.synchronize()
    assert np.array_equal(seq_d.cpu().numpy(), seq_o)
    assert np.array_equal(hist_d.cpu().numpy(), hist_o)
    assert np.array_equal(nxt.cpu().numpy(), nxt_o)
    assert np.array_equal(cu.cpu().numpy(), cu_o)
    assert np.array_equal(packed.cpu().numpy()[:cu_o[-1]], packed_o[:cu_o[-1]])
    assert np.array_equal(st.cpu().numpy(), st_o)


def test_verify_then_insert_on_device():
    """The two steps chained on one stream with no host read in between."""
    import speculative_decoding_verify_sample_gb300 as sv
    from helpers import to_device
    inp = synth.random_case(34, 64, 4, 4000, "bf16", temperature=0.8, draft_len="random",
                            greedy_frac=0.3)
    d = to_device(inp)
    L = 64
    rng = np.random.default_rng(34)
    seq = rng.integers(0, 40, size=64).astype(np.int32)
    hist = rng.integers(0, 4000, size=(64, L)).astype(np.int32)
    seq_d, hist_d = _i32(seq), _i32(hist)
    acc, out = sv.spec_verify_sample(d["target"], d["draft"], d["draft_tokens"], d["draft_len"],
                                     d["temperature"], d["uniforms"], d["uniforms_resample"])
    nxt, cu, packed, st = sv.insert_accepted(acc, out, seq_d, hist_d)
    torch.cuda.synchronize()
    acc_o, out_o, flags_o = oracle.verify_sample(inp)
    acc_h, out_h = acc.cpu().numpy(), out.cpu().numpy()
    assert_outputs_match(inp, acc_h, out_h, acc_o, out_o, flags_o, label="verify_insert")
    seq_o, hist_o, nxt_o, cu_o, packed_o, st_o = oracle.insert_accepted(acc_h, out_h, seq, hist)
    assert np.array_equal(hist_d.cpu().numpy(), hist_o) and np.array_equal(nxt.cpu().numpy(), nxt_o)
    assert np.array_equal(cu.cpu().numpy(), cu_o) and np.all(st.cpu().numpy() == 0)
