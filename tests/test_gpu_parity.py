"""CUDA path against the CPU oracle, through the C ABI (ctypes binding).

Rules (tests/helpers.py): greedy bit-exact; sampled outputs equal except at
oracle-flagged near-ties; per-row probabilities within 1e-5 relative.
"""

import numpy as np
import pytest

import oracle
from helpers import (assert_outputs_match, assert_row_stats_match, oracle_subset, report_parity,
                     run_gpu, to_device)
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


def _full_check(inp, debug=True, nthreads=8, label=None):
    acc_o, out_o, flags_o = oracle.verify_sample(inp, nthreads=nthreads)
    acc_g, out_g = run_gpu(inp)
    ties = assert_outputs_match(inp, acc_g, out_g, acc_o, out_o, flags_o, label=label)
    if debug:
        acc_d, out_d, rs = run_gpu(inp, debug=True)
        assert np.array_equal(acc_d, acc_g) and np.array_equal(out_d, out_g)
        info = oracle.row_stats(inp, nthreads=nthreads)
        assert_row_stats_match(inp, rs, info, acc_d)
    return ties


def test_tiny_sampled():
    _full_check(synth.make_inputs("tiny"), label="tiny")


def test_tiny_greedy_bit_exact():
    inp = synth.make_inputs("tiny_greedy")
    acc_o, out_o, _ = oracle.verify_sample(inp)
    acc_g, out_g = run_gpu(inp)
    assert np.array_equal(acc_g, acc_o) and np.array_equal(out_g, out_o)


RANDOM_CASES = [
    # seed, B, K, V, dtype, T, draft_len, greedy_frac
    (1, 8, 4, 1024, "f32", 1.0, None, 0.0),
    (2, 16, 3, 5000, "bf16", 0.8, "random", 0.3),
    (3, 6, 8, 70001, "bf16", 1.2, None, 0.0),        # odd V: rows not 16-byte aligned
    (4, 5, 2, 777, "f32", 0.5, None, 0.0),           # ragged last chunk
    (5, 3, 16, 3000, "f32", 1.0, "random", 0.0),     # K at the limit
    (6, 4, 1, 1, "f32", 1.0, None, 0.0),             # one-token vocabulary
    (7, 4, 2, 2, "bf16", 0.7, None, 0.5),
    (8, 10, 4, 50257, "bf16", 0.9, "random", 0.2),   # GPT-2 vocabulary
    (9, 4, 4, 300000, "bf16", 1.0, None, 0.25),      # 37 chunks per row
    (10, 3, 2, 200001, "f32", 0.6, "random", 0.0),   # unaligned f32, 49 chunks per row
    (11, 7, 5, 8, "f32", 0.3, "random", 0.3),
    (12, 2, 3, 129280, "bf16", 0.05, None, 0.0),     # small temperature
]


@pytest.mark.parametrize("seed,B,K,V,dtype,T,draft_len,greedy_frac", RANDOM_CASES)
def test_random_shapes(seed, B, K, V, dtype, T, draft_len, greedy_frac):
    inp = synth.random_case(seed, B, K, V, dtype, scale=2.0, noise=0.6, temperature=T,
                            draft_len=draft_len, greedy_frac=greedy_frac)
    _full_check(inp, label=f"random{seed}")


def test_greedy_ties_lowest_index_bf16():
    rng = np.random.default_rng(5)
    B, K, V = 64, 4, 40000
    z = rng.integers(-2, 3, size=(B, K + 1, V)).astype(np.float32)   # huge tie classes
    g = np.argmax(z, axis=2)
    x = np.where(rng.random((B, K)) < 0.7, g[:, :K], rng.integers(0, V, size=(B, K)))
    inp = dict(B=B, K=K, V=V, dtype="bf16", target=synth.bf16_bits(z), draft=None,
               draft_tokens=x.astype(np.int32), draft_len=rng.integers(1, K + 1, B).astype(np.int32),
               temperature=np.zeros(B, np.float32), uniforms=synth.uniforms24(rng, (B, K + 1)),
               uniforms_resample=synth.uniforms24(rng, (B,)))
    acc_o, out_o, _ = oracle.verify_sample(inp, nthreads=8)
    acc_g, out_g = run_gpu(inp)
    assert np.array_equal(acc_g, acc_o) and np.array_equal(out_g, out_o)


def test_unused_rows_are_not_used():
    inp = synth.random_case(21, 12, 6, 3001, "f32", temperature=1.0, draft_len="random")
    acc_ref, out_ref = run_gpu(inp)
    poisoned = dict(inp)
    tgt = inp["target"].copy()
    drf = inp["draft"].copy()
    for b, n in enumerate(inp["draft_len"]):
        tgt[b, n + 1:] = np.nan
        drf[b, n:] = np.nan
    poisoned.update(target=tgt, draft=drf)
    acc, out = run_gpu(poisoned)
    assert np.array_equal(acc, acc_ref) and np.array_equal(out, out_ref)
    acc_o, out_o, flags_o = oracle.verify_sample(poisoned)
    assert_outputs_match(poisoned, acc, out, acc_o, out_o, flags_o)


def test_all_greedy_without_draft_logits():
    inp = synth.random_case(22, 9, 3, 4099, "bf16", temperature=0.0)
    inp["draft"] = None
    acc_o, out_o, _ = oracle.verify_sample(inp)
    acc_g, out_g = run_gpu(inp)
    assert np.array_equal(acc_g, acc_o) and np.array_equal(out_g, out_o)


def test_workspace_reused_across_calls():
    import speculative_decoding_verify_sample_gb300 as sv
    ws = sv.Workspace(16, 4, 2048, "bf16", "cuda")
    a = synth.random_case(23, 16, 4, 2048, "bf16", temperature=0.9, draft_len="random",
                          greedy_frac=0.3)
    b = synth.random_case(24, 16, 4, 2048, "bf16", temperature=1.1)
    first = run_gpu(a, workspace=ws)
    run_gpu(b, workspace=ws)
    again = run_gpu(a, workspace=ws)
    assert np.array_equal(first[0], again[0]) and np.array_equal(first[1], again[1])
    assert ws.read_status() == 0


def test_device_flags_bad_data():
    import speculative_decoding_verify_sample_gb300 as sv
    inp = synth.random_case(25, 8, 3, 1000, "f32", temperature=1.0)
    inp["draft_len"] = np.array([3, 0, 4, 3, 3, 3, 3, 3], np.int32)
    inp["draft_tokens"][2, 0] = 5
    inp["draft_tokens"][3, 1] = 1000
    inp["temperature"][4] = -0.5
    inp["uniforms"][5, 2] = 1.0
    inp["target"][6, 1, :] = -np.inf         # sampled row without a finite maximum
    ws = sv.Workspace(8, 3, 1000, "f32", "cuda")
    acc, out = run_gpu(inp, workspace=ws)
    assert list(acc[[1, 2, 3, 4, 5, 6]]) == [-1] * 6
    assert np.all(out[[1, 2, 3, 4, 5, 6]] == -1)
    status = ws.read_status()
    for bit in (sv.DEV_BAD_DRAFT_LEN, sv.DEV_BAD_TOKEN, sv.DEV_BAD_TEMPERATURE,
                sv.DEV_BAD_UNIFORM, sv.DEV_BAD_ROW):
        assert status & bit, (status, bit)
    assert ws.read_status() == 0             # cleared by the read
    good = [0, 7]
    sub, acc_o, out_o, flags_o = oracle_subset(inp, good)
    assert_outputs_match(inp, acc, out, acc_o, out_o, flags_o, rows=good)


def test_sampled_request_without_draft_logits_is_flagged():
    import speculative_decoding_verify_sample_gb300 as sv
    inp = synth.random_case(26, 4, 2, 512, "f32", temperature=np.array([0, 1, 0, 0], np.float32))
    inp["draft"] = None
    ws = sv.Workspace(4, 2, 512, "f32", "cuda")
    acc, out = run_gpu(inp, workspace=ws)
    assert acc[1] == -1
    assert ws.read_status() & sv.DEV_NO_DRAFT


def test_host_entry_point_matches_device():
    import speculative_decoding_verify_sample_gb300 as sv
    inp = synth.random_case(27, 12, 4, 9000, "bf16", temperature=0.8, draft_len="random",
                            greedy_frac=0.25)
    acc_d, out_d = run_gpu(inp)
    h = {k: v.cpu().pin_memory() if v is not None else None for k, v in to_device(inp, "cpu").items()}
    staging = sv.HostStaging(12, 4, 9000, "bf16", with_draft=True, device="cuda")
    ws = sv.Workspace(12, 4, 9000, "bf16", "cuda")
    acc_h, out_h = sv.spec_verify_sample_host(h["target"], h["draft"], h["draft_tokens"],
                                              h["draft_len"], h["temperature"], h["uniforms"],
                                              h["uniforms_resample"], staging=staging, workspace=ws)
    assert np.array_equal(acc_h.numpy(), acc_d) and np.array_equal(out_h.numpy(), out_d)


@pytest.mark.parametrize("V", [7000, 7001])   # 7001: rows not 16-byte multiples (copies)
@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_host_entry_point_copies_only_read_rows(dtype, pinned, V):
    """The host entry point moves only the rows the kernels read (target
    rows t <= n_b, draft rows t < n_b of sampled requests): gathered by a
    kernel from page-locked logits, copied range by range from pageable
    ones.  The staging buffer starts as all-ones bytes (NaN logits in either
    dtype), so a read of any row it skipped would change the result; flagged
    requests (a bad draft length, a negative temperature) move no rows."""
    import torch
    import speculative_decoding_verify_sample_gb300 as sv
    B, K = 24, 6
    inp = synth.random_case(61, B, K, V, dtype, temperature=0.9, draft_len="random",
                            greedy_frac=0.3)
    inp["draft_len"][3] = K + 2          # flagged: draft length outside 1..K
    inp["temperature"][5] = -1.0         # flagged: negative temperature
    acc_d, out_d = run_gpu(inp)
    assert acc_d[3] == -1 and acc_d[5] == -1
    h = {k: (v.cpu().pin_memory() if pinned else v.cpu().contiguous()) if v is not None else None
         for k, v in to_device(inp, "cpu").items()}
    staging = sv.HostStaging(B, K, V, dtype, with_draft=True, device="cuda")
    staging.tensor.fill_(255)
    ws = sv.Workspace(B, K, V, dtype, "cuda")
    acc_h, out_h = sv.spec_verify_sample_host(h["target"], h["draft"], h["draft_tokens"],
                                              h["draft_len"], h["temperature"], h["uniforms"],
                                              h["uniforms_resample"], staging=staging, workspace=ws)
    torch.cuda.synchronize()
    assert np.array_equal(acc_h.numpy(), acc_d) and np.array_equal(out_h.numpy(), out_d)


# ---------------------------------------------------------------- full sizes


def _row_stats_check(inp, rs, acc_g, rows):
    sub, *_ = oracle_subset(inp, rows)
    info = oracle.row_stats(sub, nthreads=16)
    assert_row_stats_match(inp, rs, info, acc_g, rows=rows)


def test_llama3_full():
    inp = synth.make_inputs("llama3")
    acc_o, out_o, flags_o = oracle.verify_sample(inp, nthreads=16)
    acc_g, out_g, rs = run_gpu(inp, debug=True)
    assert_outputs_match(inp, acc_g, out_g, acc_o, out_o, flags_o, label="llama3")
    _row_stats_check(inp, rs, acc_g, np.arange(inp["B"]))


def test_greedy_full_bit_exact_with_ties_at_the_maximum():
    # N(0, 3^2) bf16 logits, nothing planted: some rows hold their maximum
    # at several indices, and the lowest must win
    inp = synth.make_inputs("greedy")
    z = synth.bf16_to_f32(inp["target"])
    tied_rows = int(((z == z.max(axis=2, keepdims=True)).sum(axis=2) > 1).sum())
    del z
    assert tied_rows >= 20
    acc_o, out_o, _ = oracle.verify_sample(inp, nthreads=16)
    acc_g, out_g, rs = run_gpu(inp, debug=True)
    assert np.array_equal(acc_g, acc_o) and np.array_equal(out_g, out_o)
    info = oracle.row_stats(inp, nthreads=16)
    assert_row_stats_match(inp, rs, info, acc_g)     # every row's argmax and maximum
    report_parity({"label": "greedy", "compared": int(inp["B"]), "sampled": 0, "excused": 0,
                   "tied_rows": tied_rows})


def test_greedy_planted_full_against_construction():
    inp = synth.make_inputs("greedy_planted")
    acc_g, out_g = run_gpu(inp)
    g = inp["planted_argmax"]
    x = inp["draft_tokens"]
    K = inp["K"]
    for b in range(inp["B"]):
        j = next((t for t in range(K) if g[b, t] != x[b, t]), K)
        assert acc_g[b] == j
        assert list(out_g[b]) == list(x[b, :j]) + [g[b, j]] + [-1] * (K - j)
    acc_o, out_o, flags_o = oracle.verify_sample(inp, nthreads=16)
    assert np.array_equal(acc_g, acc_o) and np.array_equal(out_g, out_o)


def test_dsv3_mtp_full():
    inp = synth.make_inputs("dsv3_mtp")
    acc_o, out_o, flags_o = oracle.verify_sample(inp, nthreads=16)
    acc_g, out_g, rs = run_gpu(inp, debug=True)
    assert_outputs_match(inp, acc_g, out_g, acc_o, out_o, flags_o, label="dsv3_mtp")
    _row_stats_check(inp, rs, acc_g, np.arange(0, inp["B"], 2))


def test_ragged_full():
    inp = synth.make_inputs("ragged")
    acc_o, out_o, flags_o = oracle.verify_sample(inp, nthreads=16)
    acc_g, out_g, rs = run_gpu(inp, debug=True)
    assert_outputs_match(inp, acc_g, out_g, acc_o, out_o, flags_o, label="ragged")
    _row_stats_check(inp, rs, acc_g, np.arange(0, inp["B"], 2))
    # the realised mean of emitted tokens follows the closed form per alpha
    n = inp["draft_len"]
    for a in synth.RAGGED_ALPHAS:
        sel = inp["alpha"] == a
        want = np.mean([(1 - a ** (k + 1)) / (1 - a) for k in n[sel]])
        got = (acc_g[sel] + 1).mean()
        assert abs(got - want) < 4 * max((acc_g[sel] + 1).std(), 0.5) / np.sqrt(sel.sum())


def test_constructed_near_ties_and_zero_residual():
    # requests built so that the oracle's flags are known: a zero-mass
    # residual (both sides must fall back to p), a residual of mass ~1e-3
    # drawn far from its one interior edge (no flag: must match exactly), and
    # accept ratios a little off u (flagged or not)
    rows_p, rows_q, toks, us, urs = [], [], [], [], []

    def add(zp, zq, x, u, ur):
        rows_p.append(np.asarray(zp, np.float32))
        rows_q.append(np.asarray(zq, np.float32))
        toks.append(x)
        us.append(u)
        urs.append(ur)

    V = 8
    pad = np.full(V - 3, -np.inf)
    zq0 = np.r_[0.0, 0.0, -40.0, pad]
    zp0 = np.r_[0.0, 0.0, -40.5, pad]
    for ur in (0.1, 0.3, 0.7, 0.9):                        # zero residual: draw from p
        add([zp0, np.r_[0.0, 0.0, 0.0, pad]], [zq0], [2], [0.9, 0.5], ur)
    zp1 = np.r_[np.log([0.2505, 0.2505, 0.249, 0.25]), np.full(V - 4, -np.inf)]
    zq1 = np.r_[np.zeros(4), np.full(V - 4, -np.inf)]
    for ur in (0.1, 0.25, 0.75, 0.95):                      # residual of mass ~1e-3
        add([zp1, zq1], [zq1], [2], [0.999, 0.5], ur)
    zp2 = np.r_[np.log([0.5, 0.5]), np.full(V - 2, -np.inf)]
    zq2 = np.r_[np.log([0.8, 0.2]), np.full(V - 2, -np.inf)]
    for d in (-3e-4, -5e-5, 5e-5, 3e-4):                    # accept ratio 0.625 +- d
        add([zp2, zp2], [zq2], [0], [0.625 + d, 0.3], 0.5)
    B = len(toks)
    inp = dict(B=B, K=1, V=V, dtype="f32", target=np.stack([np.stack(r) for r in rows_p]),
               draft=np.stack([np.stack(r) for r in rows_q]),
               draft_tokens=np.asarray(toks, np.int32).reshape(B, 1), draft_len=None,
               temperature=np.ones(B, np.float32),
               uniforms=np.asarray(us, np.float32).reshape(B, 2),
               uniforms_resample=np.asarray(urs, np.float32))
    acc_o, out_o, flags_o = oracle.verify_sample(inp)
    assert np.all(flags_o[:4] & oracle.RES_FALLBACK)
    assert np.all(flags_o[4:8] == 0)
    acc_g, out_g = run_gpu(inp)
    assert np.array_equal(acc_g[:8], acc_o[:8]) and np.array_equal(out_g[:8], out_o[:8])
    assert_outputs_match(inp, acc_g, out_g, acc_o, out_o, flags_o, label="constructed")


def test_batch_beyond_one_launch_sequence():
    # 2100 requests run as three launch sequences (at most 1024 requests each)
    # sharing one workspace: each must leave its draw lists empty for the next
    inp = synth.random_case(31, 2100, 3, 700, "bf16", temperature=0.9, draft_len="random",
                            greedy_frac=0.3)
    _full_check(inp)


@pytest.mark.parametrize("greedy_frac", [0.0, 1.0])
def test_records_beyond_decide_staging(greedy_frac):
    # K = 16 and 98 chunks per row: 33 rows x 98 records exceed the 2048
    # records a decide CTA stages at once, so its warps combine a row each
    inp = synth.random_case(32, 3, 16, 300000, "bf16", temperature=1.0, greedy_frac=greedy_frac)
    _full_check(inp)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_vocabulary_at_the_row_limit(dtype):
    import speculative_decoding_verify_sample_gb300 as sv
    V = sv.max_vocab(dtype)   # 2 MB rows
    inp = synth.random_case(33, 2, 2, V, dtype, temperature=1.0, draft_len=[2, 1])
    _full_check(inp)
