"""The C ABI without a GPU: the library builds, loads, exports every function
include/specverify.h declares, and rejects bad host-side arguments before
touching the device."""

import ctypes
import os
import re

import pytest

import speculative_decoding_verify_sample_gb300 as sv
from speculative_decoding_verify_sample_gb300 import _native

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "specverify.h")


@pytest.fixture(scope="module")
def L():
    sv.build()
    return sv.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spec\w+)\s*\(", text)))


def declared_arity():
    """Parameter count of every function the header declares."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {}
    for name, params in re.findall(r"\b(spec\w+)\s*\(([^;{]*?)\)\s*;", text):
        params = params.strip()
        out[name] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_signatures_match_the_header():
    """The ctypes table passes exactly the arguments each C function takes."""
    arity = declared_arity()
    assert arity, "no declarations parsed"
    for name, n in arity.items():
        assert name in _native.SIGNATURES, name
        assert len(_native.SIGNATURES[name][1]) == n, (name, n, len(_native.SIGNATURES[name][1]))


def test_header_declares_expected_entry_points():
    names = declared_functions()
    for must in ("spec_verify_sample", "spec_verify_sample_debug", "spec_verify_sample_host",
                 "specv_workspace_bytes", "specv_workspace_init", "specv_read_device_status"):
        assert must in names


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), name
        assert name in _native.SIGNATURES, f"binding lacks {name}"


def test_limits_and_sizes(L):
    assert L.specv_max_vocab(0) >= 262144
    assert L.specv_max_vocab(1) >= 262144
    assert L.specv_max_vocab(7) == 0
    assert L.specv_workspace_bytes(0, 4, 1000, 1) == 0
    assert L.specv_workspace_bytes(4, 17, 1000, 1) == 0
    assert L.specv_workspace_bytes(4, 4, 0, 1) == 0
    assert L.specv_workspace_bytes(4, 4, 1000, 5) == 0
    assert L.specv_workspace_bytes(4, 4, L.specv_max_vocab(1) + 1, 1) == 0
    # at least one 8-byte record per (request, row, chunk of at most 16 KB)
    assert L.specv_workspace_bytes(32, 4, 128256, 1) >= 32 * 9 * 16 * 8
    assert L.specv_workspace_bytes(32, 4, 128256, 0) > L.specv_workspace_bytes(32, 4, 128256, 1)
    assert L.specv_host_staging_bytes(2, 2, 100, 1, 1) >= 2 * 3 * 100 * 2 + 2 * 2 * 100 * 2
    assert L.specv_status_string(0) == b"ok"


FAKE = 0x10000  # a 64 KB-aligned non-null address: host checks never dereference it


def _call(L, **over):
    a = dict(target=FAKE, draft=FAKE, dtype=1, tokens=FAKE, dlen=FAKE, temp=FAKE, uni=FAKE,
             ures=FAKE, B=4, K=4, V=1024, acc=FAKE, out=FAKE, ws=FAKE, wsb=1 << 20)
    a.update(over)
    return L.spec_verify_sample(a["target"], a["draft"], a["dtype"], a["tokens"], a["dlen"],
                                a["temp"], a["uni"], a["ures"], a["B"], a["K"], a["V"], a["acc"],
                                a["out"], a["ws"], a["wsb"], None)


@pytest.mark.parametrize("over,status", [
    (dict(target=None), 1), (dict(tokens=None), 1), (dict(acc=None), 1), (dict(ws=None), 1),
    (dict(dtype=3), 1), (dict(B=0), 1), (dict(K=0), 1), (dict(V=0), 1),
    (dict(K=17), 2), (dict(B=70000), 2), (dict(V=1048577), 2), (dict(dtype=0, V=524289), 2),
    (dict(wsb=8), 3), (dict(target=FAKE + 1), 1), (dict(ws=FAKE + 128), 1), (dict(uni=FAKE + 2), 1),
])
def test_host_side_argument_errors(L, over, status):
    assert _call(L, **over) == status


def test_debug_entry_requires_row_stats(L):
    rc = L.spec_verify_sample_debug(FAKE, FAKE, 1, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 4, 1024, FAKE,
                                    FAKE, FAKE, 1 << 20, None, None)
    assert rc == 1


def test_host_entry_rejects_small_staging(L):
    rc = L.spec_verify_sample_host(FAKE, FAKE, 1, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 4, 1024, FAKE,
                                   FAKE, FAKE, 64, FAKE, 1 << 20, None)
    assert rc == 3


def test_binding_refuses_cpu_tensors():
    torch = pytest.importorskip("torch")
    t = torch.zeros(2, 3, 8)
    with pytest.raises(ValueError):
        sv.spec_verify_sample(t, None, torch.zeros(2, 2, dtype=torch.int32), None,
                              torch.zeros(2), torch.zeros(2, 3), torch.zeros(2))


def test_noalloc_rejects_shapes_beyond_its_array(L):
    # the size check runs on the host before any pointer is used
    B, K, V = 1024, 16, 500000
    assert L.specv_workspace_bytes(B, K, V, 1) > _native.NOALLOC_SCRATCH_BYTES
    rc = L.spec_verify_sample_noalloc(FAKE, FAKE, 1, FAKE, FAKE, FAKE, FAKE, FAKE, B, K, V, FAKE,
                                      FAKE, None)
    assert rc == 2


def test_new_entry_points_reject_bad_host_arguments(L):
    # draft-side sampler: null logits, zero rows, a too-small workspace
    assert L.spec_sample_draft(None, 1, FAKE, FAKE, 4, 100, FAKE, FAKE, 1 << 20, None, None) == 1
    assert L.spec_sample_draft(FAKE, 1, FAKE, FAKE, 0, 100, FAKE, FAKE, 1 << 20, None, None) == 1
    assert L.spec_sample_draft(FAKE, 1, FAKE, FAKE, 4, 100, FAKE, FAKE, 8, None, None) == 3
    assert L.specv_sample_workspace_bytes(4, 100, 1) > 0
    assert L.specv_sample_workspace_bytes(0, 100, 1) == 0
    # one-hot rule: no resample uniforms, K beyond the limit
    assert L.spec_verify_sample_onehot(FAKE, 1, FAKE, FAKE, FAKE, FAKE, None, 4, 4, 100, FAKE,
                                       FAKE, FAKE, 1 << 20, None, None) == 1
    assert L.spec_verify_sample_onehot(FAKE, 1, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 17, 100, FAKE,
                                       FAKE, FAKE, 1 << 20, None, None) == 2
    # tree: N beyond 64 nodes, no parents, workspace sizing
    assert L.specv_tree_workspace_bytes(4, 65, 100, 1) == 0
    assert L.specv_tree_workspace_bytes(4, 64, 100, 1) > 0
    assert L.spec_verify_tree_greedy(FAKE, 1, FAKE, FAKE, FAKE, 4, 65, 100, FAKE, FAKE, FAKE, FAKE,
                                     1 << 24, None, None) == 2
    assert L.spec_verify_tree_greedy(FAKE, 1, None, FAKE, FAKE, 4, 8, 100, FAKE, FAKE, FAKE, FAKE,
                                     1 << 24, None, None) == 1
    # insert: null buffers, misaligned history
    assert L.spec_insert_accepted(None, FAKE, 4, 2, FAKE, FAKE, 16, FAKE, FAKE, FAKE, FAKE, None) == 1
    assert L.spec_insert_accepted(FAKE, FAKE, 4, 2, FAKE, FAKE + 2, 16, FAKE, FAKE, FAKE, FAKE,
                                  None) == 1
