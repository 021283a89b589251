"""Shared test helpers: moving synthetic inputs to the GPU and comparing the
CUDA path with the oracle under the parity rules.

Parity rules (fixed for this sampler):
  * greedy requests (T = 0): accepted_len and out_tokens bit-exact;
  * sampled requests: accepted_len and out_tokens equal, except where the
    oracle flags a near-tie: |u - p/q| < 1e-4 at an evaluated position, the
    final draw's target u*W within 1e-4*W of an edge of its CDF bucket, or
    within 2e-5 of probability mass of such an edge (the shift a 1e-5
    relative error on every p_i and q_i can cause), or a residual of exactly
    zero mass.  Excused mismatches are counted per flag, reported, and held
    under a ceiling;
  * per-row statistics: max logits exact; S_p, S_q within 1e-5 relative;
    ln p(x_t), ln q(x_t) within 1e-5 absolute (1e-5 relative on p, q); at
    the final row (t = accepted_len) the final-draw mass within 1e-5
    absolute and the drawn token equal except at flagged rows; at T = 0 the
    argmax of every row bit-exact.
"""

from __future__ import annotations

import numpy as np

import oracle

PROB_RTOL = 1e-5
MASS_ATOL = 1e-5


def to_device(inp, device="cuda"):
    import torch

    def logits(a):
        if a is None:
            return None
        if inp["dtype"] == "bf16":
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(device)

    def i32(a):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(device)

    def f32(a):
        return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(device)

    return dict(target=logits(inp["target"]), draft=logits(inp.get("draft")),
                draft_tokens=i32(inp["draft_tokens"]), draft_len=i32(inp.get("draft_len")),
                temperature=f32(inp["temperature"]), uniforms=f32(inp["uniforms"]),
                uniforms_resample=f32(inp["uniforms_resample"]))


def run_gpu(inp, debug=False, workspace=None, device="cuda"):
    import torch
    import speculative_decoding_verify_sample_gb300 as sv
    d = to_device(inp, device)
    args = (d["target"], d["draft"], d["draft_tokens"], d["draft_len"], d["temperature"],
            d["uniforms"], d["uniforms_resample"])
    if debug:
        acc, out, rs = sv.spec_verify_sample_debug(*args, workspace=workspace)
        torch.cuda.synchronize()
        return acc.cpu().numpy(), out.cpu().numpy(), rs.cpu().numpy()
    acc, out = sv.spec_verify_sample(*args, workspace=workspace)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), out.cpu().numpy()


def excuse_ceiling(n_sampled: int) -> int:
    """Most excused (flagged near-tie) mismatches a comparison may have: a
    near-tie band of width ~1e-4 is hit by well under 1% of requests."""
    return max(3, int(np.ceil(0.01 * n_sampled)))


def assert_outputs_match(inp, acc_g, out_g, acc_o, out_o, flags_o, rows=None, label=None):
    """Checks the parity rules; returns the excused-mismatch report: counts
    of mismatched requests by oracle flag, the requests flagged, and the
    total compared (also printed and appended to $SPECV_PARITY_LOG)."""
    idx = np.arange(inp["B"]) if rows is None else np.asarray(rows)
    T = np.asarray(inp["temperature"])[idx]
    mism = (acc_g[idx] != acc_o) | np.any(out_g[idx] != out_o, axis=1)
    greedy_bad = mism & (T == 0)
    assert not greedy_bad.any(), (
        f"greedy mismatch at requests {idx[greedy_bad][:8]}: gpu {acc_g[idx][greedy_bad][:4]} "
        f"{out_g[idx][greedy_bad][:4]} oracle {acc_o[greedy_bad][:4]} {out_o[greedy_bad][:4]}")
    allowed = (flags_o & oracle.NEAR_TIE_MASK) != 0
    bad = mism & ~allowed
    assert not bad.any(), (
        f"unflagged mismatch at requests {idx[bad][:8]}: gpu acc {acc_g[idx][bad][:4]} "
        f"out {out_g[idx][bad][:4]} / oracle acc {acc_o[bad][:4]} out {out_o[bad][:4]} "
        f"flags {flags_o[bad][:4]}")
    excused = mism & allowed
    report = {"label": label, "compared": int(len(idx)), "sampled": int((T > 0).sum()),
              "excused": int(excused.sum()),
              "flagged": {name: int(((flags_o & bit) != 0).sum())
                          for bit, name in oracle.FLAG_NAMES.items()},
              "excused_by_flag": {name: int((excused & ((flags_o & bit) != 0)).sum())
                                  for bit, name in oracle.FLAG_NAMES.items()}}
    report_parity(report)
    assert report["excused"] <= excuse_ceiling(report["sampled"]), report
    return report


def report_parity(report):
    """Prints one parity report and appends it to $SPECV_PARITY_LOG (JSON lines)."""
    import json
    import os
    line = json.dumps(report)
    print("parity", line)
    path = os.environ.get("SPECV_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(line + "\n")


def assert_row_stats_match(inp, rs_g, info_o, acc_g, rows=None):
    """Per-row statistics of the debug entry point against the oracle.
    acc_g: the GPU's accepted lengths (the final draw sits at row acc_g[b])."""
    idx = np.arange(inp["B"]) if rows is None else np.asarray(rows)
    K = inp["K"]
    n_all = np.full(inp["B"], K) if inp.get("draft_len") is None else np.asarray(inp["draft_len"])
    T_all = np.asarray(inp["temperature"])
    flagged_rows = 0
    for r, b in enumerate(idx):
        n, T = int(n_all[b]), float(T_all[b])
        for t in range(n + 1):
            g = rs_g[b, t].astype(np.float64)
            o = info_o[r, t]
            assert g[0] == o[0], (b, t, "max_p", g[0], o[0])
            if T == 0:
                assert g[7] == o[7], (b, t, "argmax", g[7], o[7])
                continue
            assert abs(g[1] - o[1]) <= PROB_RTOL * o[1], (b, t, "S_p", g[1], o[1])
            if t < n:
                assert g[3] == o[3], (b, t, "max_q", g[3], o[3])
                assert abs(g[4] - o[4]) <= PROB_RTOL * o[4], (b, t, "S_q", g[4], o[4])
                assert abs(g[2] - o[2]) <= PROB_RTOL, (b, t, "ln p(x)", g[2], o[2])
                assert abs(g[5] - o[5]) <= PROB_RTOL, (b, t, "ln q(x)", g[5], o[5])
            if t != acc_g[b]:
                continue
            assert abs(g[6] - o[6]) <= MASS_ATOL, (b, t, "mass", g[6], o[6])
            row_flag = o[8] != 0   # the draw's own CDF-edge or zero-residual flag
            if g[7] != o[7]:
                assert row_flag, (b, t, "candidate", g[7], o[7], "mass", o[6])
                flagged_rows += 1
    return flagged_rows


def oracle_subset(inp, rows, nthreads=8):
    """The oracle on a subset of requests (same arrays, sliced)."""
    rows = np.asarray(rows)
    sub = dict(inp)
    sub["B"] = len(rows)
    for k in ("target", "draft", "draft_tokens", "draft_len", "temperature", "uniforms",
              "uniforms_resample"):
        if sub.get(k) is not None:
            sub[k] = np.ascontiguousarray(np.asarray(inp[k])[rows])
    acc, out, flags = oracle.verify_sample(sub, nthreads=nthreads)
    return sub, acc, out, flags
