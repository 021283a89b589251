"""CPU oracle for the speculative-decoding verification sampler.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check and
the benchmark's CPU-baseline leg may import this package.  The oracle is plain
C++ in double precision (``specverify_oracle.cpp``); this module compiles it
with the host compiler and calls it through ctypes.  It shares no code with the
CUDA library.

Rule followed: "Decodificación Especulativa y EAGLE" (Phase 10 - Lesson 25),
sections "La Regla de Exactitud" and "Caso codicioso"; the n+1 bound from
"Accelerating Sonar through speculation", section "Decodificación especulativa".
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "specverify_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

# near-tie / condition flags (bitmask per request)
TIE_ACCEPT = 1       # |u - p/q| < 1e-4 at an evaluated position
TIE_CDF = 2          # the final draw's u*W lies within 1e-4*W of an edge of its bucket
PRECISION_BAND = 4   # ... within EDGE_ABS of such an edge (not within 1e-4*W)
RES_FALLBACK = 8     # residual mass exactly 0: the replacement was drawn from p
BAD_INPUT = 16       # the request was rejected as invalid
NEAR_TIE_MASK = TIE_ACCEPT | TIE_CDF | PRECISION_BAND | RES_FALLBACK
FLAG_NAMES = {TIE_ACCEPT: "tie_accept", TIE_CDF: "tie_cdf", PRECISION_BAND: "precision_band",
              RES_FALLBACK: "res_fallback"}

TIE_BAND = 1e-4      # relative band of the accept test and of a CDF edge (times W)
EDGE_ABS = 2e-5      # absolute floor of the CDF-edge band, in probability mass

ROW_INFO = 10        # doubles per row in row_stats()

DTYPES = {"f32": 0, "bf16": 1}


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/liboracle.so`` (host compiler only)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            vp, i32p, f32p = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
            lib.oracle_verify_sample.argtypes = [vp, vp, ctypes.c_int, i32p, i32p, f32p, f32p, f32p,
                                                 ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                 i32p, i32p, i32p, ctypes.c_int]
            lib.oracle_verify_sample.restype = ctypes.c_int
            lib.oracle_row_stats.argtypes = [vp, vp, ctypes.c_int, i32p, i32p, f32p, f32p, f32p,
                                             ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, ctypes.c_int]
            lib.oracle_row_stats.restype = ctypes.c_int
            lib.oracle_version.restype = ctypes.c_int
            lib.oracle_sample_draft.argtypes = [vp, ctypes.c_int, f32p, f32p, ctypes.c_int,
                                                ctypes.c_int, i32p, i32p, ctypes.c_int]
            lib.oracle_sample_draft.restype = ctypes.c_int
            lib.oracle_verify_onehot.argtypes = [vp, ctypes.c_int, i32p, i32p, f32p, f32p, f32p,
                                                 ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                 i32p, i32p, i32p, ctypes.c_int]
            lib.oracle_verify_onehot.restype = ctypes.c_int
            lib.oracle_tree_greedy.argtypes = [vp, ctypes.c_int, i32p, i32p, i32p, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int, i32p, i32p, i32p,
                                               ctypes.c_int]
            lib.oracle_tree_greedy.restype = ctypes.c_int
            lib.oracle_insert_accepted.argtypes = [i32p, i32p, ctypes.c_int, ctypes.c_int, i32p,
                                                   i32p, ctypes.c_int, i32p, i32p, i32p, i32p]
            lib.oracle_insert_accepted.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _prep(inp):
    dt = inp["dtype"]
    want = np.uint16 if dt == "bf16" else np.float32
    tgt = np.ascontiguousarray(inp["target"], dtype=want)
    drf = None if inp.get("draft") is None else np.ascontiguousarray(inp["draft"], dtype=want)
    toks = np.ascontiguousarray(inp["draft_tokens"], dtype=np.int32)
    dl = None if inp.get("draft_len") is None else np.ascontiguousarray(inp["draft_len"], dtype=np.int32)
    temp = np.ascontiguousarray(inp["temperature"], dtype=np.float32)
    uni = np.ascontiguousarray(inp["uniforms"], dtype=np.float32)
    ur = np.ascontiguousarray(inp["uniforms_resample"], dtype=np.float32)
    B, K, V = int(inp["B"]), int(inp["K"]), int(inp["V"])
    assert tgt.size == B * (K + 1) * V, "target logits must be [B, K+1, V]"
    assert drf is None or drf.size == B * K * V, "draft logits must be [B, K, V]"
    assert toks.size == B * K and temp.size == B and uni.size == B * (K + 1) and ur.size == B
    return tgt, drf, DTYPES[dt], toks, dl, temp, uni, ur, B, K, V


def verify_sample(inp, nthreads: int = 1):
    """Run the rule on host arrays.

    ``inp`` holds numpy arrays ``target`` [B,K+1,V], ``draft`` [B,K,V] (bf16 as
    raw uint16, or float32), ``draft_tokens`` [B,K], ``draft_len`` [B] (or None),
    ``temperature`` [B], ``uniforms`` [B,K+1], ``uniforms_resample`` [B], plus
    ``dtype`` ("f32"/"bf16") and B, K, V.  Returns (accepted_len [B],
    out_tokens [B,K+1], flags [B]).
    """
    lib = _load()
    tgt, drf, dt, toks, dl, temp, uni, ur, B, K, V = _prep(inp)
    acc = np.empty(B, np.int32)
    out = np.empty((B, K + 1), np.int32)
    flags = np.empty(B, np.int32)
    rc = lib.oracle_verify_sample(_ptr(tgt), _ptr(drf), dt, _ptr(toks), _ptr(dl), _ptr(temp),
                                  _ptr(uni), _ptr(ur), B, K, V, _ptr(acc), _ptr(out), _ptr(flags),
                                  int(nthreads))
    if rc != 0:
        raise ValueError("oracle_verify_sample rejected its arguments")
    return acc, out, flags


def row_stats(inp, nthreads: int = 1):
    """Per-row quantities, float64 array [B, K+1, 10]:
    zmax_p, S_p, log p(x_t), zmax_q, S_q, log q(x_t), W, candidate token,
    the candidate draw's flags (TIE_CDF, PRECISION_BAND, RES_FALLBACK bits),
    accept-test near-tie flag (NaN where a row is unused)."""
    lib = _load()
    tgt, drf, dt, toks, dl, temp, uni, ur, B, K, V = _prep(inp)
    info = np.empty((B, K + 1, ROW_INFO), np.float64)
    rc = lib.oracle_row_stats(_ptr(tgt), _ptr(drf), dt, _ptr(toks), _ptr(dl), _ptr(temp),
                              _ptr(uni), _ptr(ur), B, K, V, _ptr(info), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_row_stats rejected its arguments")
    return info


def _logits(a, dtype):
    return np.ascontiguousarray(a, dtype=np.uint16 if dtype == "bf16" else np.float32)


def sample_draft(logits, dtype, temperature, uniforms, nthreads: int = 1):
    """The draft-side sampler ("Decodificación Especulativa y EAGLE", sections
    "La Configuración de Dos Modelos", "Desarrolla"): one token per row of
    ``logits`` [R, V] from softmax(z / T) by inverse CDF with ``uniforms``
    [R]; the row's lowest-index argmax at T = 0.  Returns (tokens [R],
    flags [R]) int32 (flags: TIE_CDF / PRECISION_BAND near-ties, BAD_INPUT)."""
    lib = _load()
    z = _logits(logits, dtype)
    R, V = z.shape
    T = np.ascontiguousarray(temperature, np.float32)
    u = np.ascontiguousarray(uniforms, np.float32)
    assert T.size == R and u.size == R
    tok = np.empty(R, np.int32)
    flags = np.empty(R, np.int32)
    rc = lib.oracle_sample_draft(_ptr(z), DTYPES[dtype], _ptr(T), _ptr(u), R, V, _ptr(tok),
                                 _ptr(flags), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_sample_draft rejected its arguments")
    return tok, flags


def verify_onehot(inp, nthreads: int = 1):
    """The verification rule for a draft that proposes its top token (q is
    the point mass at the drafted token; ``inp`` as for verify_sample, draft
    logits unused).  Returns (accepted_len [B], out_tokens [B,K+1], flags [B])."""
    lib = _load()
    tgt, _, dt, toks, dl, temp, uni, ur, B, K, V = _prep(dict(inp, draft=None))
    acc = np.empty(B, np.int32)
    out = np.empty((B, K + 1), np.int32)
    flags = np.empty(B, np.int32)
    rc = lib.oracle_verify_onehot(_ptr(tgt), dt, _ptr(toks), _ptr(dl), _ptr(temp), _ptr(uni),
                                  _ptr(ur), B, K, V, _ptr(acc), _ptr(out), _ptr(flags),
                                  int(nthreads))
    if rc != 0:
        raise ValueError("oracle_verify_onehot rejected its arguments")
    return acc, out, flags


def tree_greedy(target, dtype, parents, tokens, n_nodes, nthreads: int = 1):
    """Greedy verification of a token tree ("Decodificación Especulativa y
    EAGLE", section "Verificación de Atención en Árvore"): ``target`` [B, N, V]
    logits per tree node, ``parents`` [B, N] (-1 at the root, else < i),
    ``tokens`` [B, N], ``n_nodes`` [B].  Returns (accepted_len [B],
    out_tokens [B, N], path_nodes [B, N]) int32."""
    lib = _load()
    z = _logits(target, dtype)
    B, N, V = z.shape
    par = np.ascontiguousarray(parents, np.int32).reshape(B, N)
    tok = np.ascontiguousarray(tokens, np.int32).reshape(B, N)
    nn = np.ascontiguousarray(n_nodes, np.int32).reshape(B)
    acc = np.empty(B, np.int32)
    out = np.empty((B, N), np.int32)
    path = np.empty((B, N), np.int32)
    rc = lib.oracle_tree_greedy(_ptr(z), DTYPES[dtype], _ptr(par), _ptr(tok), _ptr(nn), B, N, V,
                                _ptr(acc), _ptr(out), _ptr(path), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_tree_greedy rejected its arguments")
    return acc, out, path


def insert_accepted(accepted_len, out_tokens, seq_lens, history):
    """The post-accept insert ("Accelerating Sonar through speculation",
    section "Programación MTP para un solo token").  Returns (seq_lens [B],
    history [B, L], next_tokens [B], cu_emitted [B+1], packed [B*(K+1)],
    status [B]); the inputs are not modified."""
    lib = _load()
    acc = np.ascontiguousarray(accepted_len, np.int32)
    out = np.ascontiguousarray(out_tokens, np.int32)
    B, K1 = out.shape
    seq = np.array(seq_lens, np.int32, copy=True)
    hist = np.array(history, np.int32, copy=True)
    L = hist.shape[1]
    nxt = np.empty(B, np.int32)
    cu = np.empty(B + 1, np.int32)
    packed = np.full(B * K1, -1, np.int32)
    status = np.empty(B, np.int32)
    rc = lib.oracle_insert_accepted(_ptr(acc), _ptr(out), B, K1, _ptr(seq), _ptr(hist), L,
                                    _ptr(nxt), _ptr(cu), _ptr(packed), _ptr(status))
    if rc != 0:
        raise ValueError("oracle_insert_accepted rejected its arguments")
    return seq, hist, nxt, cu, packed, status
