"""GB300-native speculative-decoding verification sampler.

The sampler ("Decodificación Especulativa y EAGLE", Phase 10 - Lesson 25,
sections "La Regla de Exactitud" and "Caso codicioso") runs as hand-written
CUDA for sm_103a behind the C ABI in include/specverify.h.  This module is the
thin Python binding: it checks shapes and dtypes of torch tensors, passes
their device pointers and the current CUDA stream to the library, and turns
status codes into exceptions.  Nothing here computes any step of the rule.
"""

from __future__ import annotations

from ._native import (DEV_BAD_DRAFT_LEN, DEV_BAD_ROW, DEV_BAD_TEMPERATURE, DEV_BAD_TOKEN,
                      DEV_BAD_TREE, DEV_BAD_UNIFORM, DEV_NO_DRAFT, DEV_TIMEOUT, SPECV_BF16,
                      SPECV_F32, SpecVerifyError, check, lib)
from .build import build

__all__ = [
    "build", "lib", "Workspace", "HostStaging", "spec_verify_sample", "spec_verify_sample_debug",
    "spec_verify_sample_host", "spec_verify_sample_noalloc", "sample_draft",
    "spec_verify_sample_onehot", "verify_tree_greedy", "insert_accepted", "launch_plan",
    "workspace_bytes", "max_vocab", "SpecVerifyError", "DEV_BAD_TREE",
    "DEV_BAD_DRAFT_LEN", "DEV_BAD_TOKEN", "DEV_BAD_TEMPERATURE", "DEV_BAD_UNIFORM",
    "DEV_BAD_ROW", "DEV_NO_DRAFT", "DEV_TIMEOUT",
]


def _torch():
    import torch
    return torch


def _stream_ptr(stream, device):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dtype_code(t):
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return SPECV_BF16
    if t.dtype == torch.float32:
        return SPECV_F32
    raise TypeError(f"logits must be bfloat16 or float32, got {t.dtype}")


def _code(dtype):
    torch = _torch()
    return SPECV_BF16 if dtype in (torch.bfloat16, "bf16", SPECV_BF16) else SPECV_F32


def workspace_bytes(B: int, K: int, V: int, dtype) -> int:
    """Device workspace bytes spec_verify_sample needs for these sizes (0:
    out of range)."""
    return int(lib().specv_workspace_bytes(B, K, V, _code(dtype)))


def launch_plan(B: int, K: int, V: int, dtype, with_draft: bool = True) -> dict:
    """The launch shape the library picks for these sizes (needs a GPU)."""
    import ctypes
    torch = _torch()
    code = SPECV_BF16 if dtype in (torch.bfloat16, "bf16") else SPECV_F32
    out = (ctypes.c_int32 * 6)()
    check("specv_launch_plan", lib().specv_launch_plan(B, K, V, code, int(with_draft), out))
    return dict(ctas=out[0], chunk=out[1], slots_per_warp=out[2], chunks_per_row=out[3], smem=out[4],
                threads=out[5])


def max_vocab(dtype) -> int:
    """The largest vocabulary the library takes for this dtype (2 MB rows)."""
    torch = _torch()
    code = SPECV_BF16 if dtype in (torch.bfloat16, "bf16") else SPECV_F32
    return int(lib().specv_max_vocab(code))


class Workspace:
    """Device workspace for calls over B requests of up to K drafts of a
    V-entry vocabulary, zeroed once on creation (every call leaves it ready
    for the next).  kind "sample": B rows for sample_draft (K unused);
    kind "tree": B trees of up to K nodes for verify_tree_greedy."""

    def __init__(self, B: int, K: int, V: int, dtype, device=None, stream=None, kind="verify"):
        torch = _torch()
        if kind == "sample":
            n = int(lib().specv_sample_workspace_bytes(B, V, _code(dtype)))
        elif kind == "tree":
            n = int(lib().specv_tree_workspace_bytes(B, K, V, _code(dtype)))
        else:
            n = workspace_bytes(B, K, V, dtype)
        if n == 0:
            raise ValueError(f"unsupported workspace shape B={B} K={K} V={V}")
        self.B, self.K, self.V, self.nbytes = B, K, V, n
        self.tensor = torch.empty(n, dtype=torch.uint8, device=device)
        check("specv_workspace_init",
              lib().specv_workspace_init(self.tensor.data_ptr(), n,
                                         _stream_ptr(stream, self.tensor.device)))

    def read_status(self, stream=None) -> int:
        """Device status word (bits DEV_*); synchronises the stream and clears it."""
        out = __import__("ctypes").c_int32(0)
        lib().specv_read_device_status(self.tensor.data_ptr(), self.nbytes,
                                       __import__("ctypes").byref(out),
                                       _stream_ptr(stream, self.tensor.device))
        return int(out.value)


def _check_inputs(target, draft, draft_tokens, draft_len, temperature, uniforms, uniforms_resample):
    torch = _torch()
    if target.dim() != 3:
        raise ValueError("target_logits must be [B, K+1, V]")
    B, K1, V = target.shape
    K = K1 - 1
    if K < 1:
        raise ValueError("target_logits needs K+1 >= 2 positions")
    dev = target.device
    if dev.type != "cuda":
        raise ValueError("spec_verify_sample takes CUDA tensors (use spec_verify_sample_host)")

    def need(name, t, shape, dtype):
        if t is None:
            return
        if tuple(t.shape) != tuple(shape):
            raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
        if t.dtype != dtype:
            raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
        if t.device != dev:
            raise ValueError(f"{name} is on {t.device}, target_logits on {dev}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")

    need("target_logits", target, (B, K + 1, V), target.dtype)
    _dtype_code(target)
    need("draft_logits", draft, (B, K, V), target.dtype)
    need("draft_tokens", draft_tokens, (B, K), torch.int32)
    need("draft_len", draft_len, (B,), torch.int32)
    need("temperature", temperature, (B,), torch.float32)
    need("uniforms", uniforms, (B, K + 1), torch.float32)
    need("uniforms_resample", uniforms_resample, (B,), torch.float32)
    return B, K, V


def _ptr(t):
    return None if t is None else t.data_ptr()


def _run(fn_name, target, draft, draft_tokens, draft_len, temperature, uniforms, uniforms_resample,
         workspace, accepted_len, out_tokens, stream, row_stats):
    torch = _torch()
    B, K, V = _check_inputs(target, draft, draft_tokens, draft_len, temperature, uniforms,
                            uniforms_resample)
    dev = target.device
    if accepted_len is None:
        accepted_len = torch.empty(B, dtype=torch.int32, device=dev)
    if out_tokens is None:
        out_tokens = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = Workspace(B, K, V, target.dtype, dev, stream)
    args = [_ptr(target), _ptr(draft), _dtype_code(target), _ptr(draft_tokens), _ptr(draft_len),
            _ptr(temperature), _ptr(uniforms), _ptr(uniforms_resample), B, K, V,
            _ptr(accepted_len), _ptr(out_tokens), workspace.tensor.data_ptr(), workspace.nbytes]
    if row_stats is not None:
        args.append(_ptr(row_stats))
    with torch.cuda.device(dev):   # the library works on the current device
        args.append(_stream_ptr(stream, dev))
        check(fn_name, getattr(lib(), fn_name)(*args))
    return accepted_len, out_tokens


def spec_verify_sample(target_logits, draft_logits, draft_tokens, draft_len, temperature, uniforms,
                       uniforms_resample, *, workspace=None, accepted_len=None, out_tokens=None,
                       stream=None):
    """Verify drafted tokens on the GPU.  Tensors on one CUDA device:
    target_logits [B,K+1,V] bf16/f32, draft_logits [B,K,V] same dtype (or None
    when every temperature is 0), draft_tokens [B,K] int32, draft_len [B]
    int32 (or None = all K), temperature [B] f32 (0 = greedy), uniforms
    [B,K+1] f32, uniforms_resample [B] f32.  Returns (accepted_len [B],
    out_tokens [B,K+1]) int32; asynchronous on the current stream."""
    return _run("spec_verify_sample", target_logits, draft_logits, draft_tokens, draft_len,
                temperature, uniforms, uniforms_resample, workspace, accepted_len, out_tokens,
                stream, None)


def spec_verify_sample_debug(target_logits, draft_logits, draft_tokens, draft_len, temperature,
                             uniforms, uniforms_resample, *, workspace=None, accepted_len=None,
                             out_tokens=None, row_stats=None, stream=None):
    """As spec_verify_sample, plus per-row statistics [B, K+1, 8] float32
    (max_p, S_p, ln p(x), max_q, S_q, ln q(x), final-draw mass, drawn token;
    the last two at the final row only); unused slots are left as NaN."""
    torch = _torch()
    B, K1, _ = target_logits.shape
    if row_stats is None:
        row_stats = torch.full((B, K1, 8), float("nan"), dtype=torch.float32,
                               device=target_logits.device)
    acc, out = _run("spec_verify_sample_debug", target_logits, draft_logits, draft_tokens,
                    draft_len, temperature, uniforms, uniforms_resample, workspace, accepted_len,
                    out_tokens, stream, row_stats)
    return acc, out, row_stats


class HostStaging:
    """Device staging buffer for spec_verify_sample_host."""

    def __init__(self, B: int, K: int, V: int, dtype, with_draft: bool = True, device=None):
        torch = _torch()
        code = SPECV_BF16 if dtype in (torch.bfloat16, "bf16") else SPECV_F32
        n = int(lib().specv_host_staging_bytes(B, K, V, code, int(with_draft)))
        if n == 0:
            raise ValueError("unsupported staging shape")
        self.nbytes = n
        self.tensor = torch.empty(n, dtype=torch.uint8, device=device)


def spec_verify_sample_host(target_logits, draft_logits, draft_tokens, draft_len, temperature,
                            uniforms, uniforms_resample, *, staging, workspace, accepted_len=None,
                            out_tokens=None, stream=None):
    """The sampler on host (CPU, ideally pinned) tensors: the library moves
    the logit rows the rule reads to the device (gathered by a kernel from
    pinned tensors, copied range by range from pageable ones) with the small
    inputs, runs, copies the outputs back and synchronises."""
    torch = _torch()
    if target_logits.device.type != "cpu":
        raise ValueError("spec_verify_sample_host takes host tensors")
    B, K1, V = target_logits.shape
    K = K1 - 1
    for name, t in (("target_logits", target_logits), ("draft_logits", draft_logits),
                    ("draft_tokens", draft_tokens), ("draft_len", draft_len),
                    ("temperature", temperature), ("uniforms", uniforms),
                    ("uniforms_resample", uniforms_resample)):
        if t is not None and (t.device.type != "cpu" or not t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous host tensor")
    if accepted_len is None:
        accepted_len = torch.empty(B, dtype=torch.int32).pin_memory()
    if out_tokens is None:
        out_tokens = torch.empty((B, K + 1), dtype=torch.int32).pin_memory()
    dev = staging.tensor.device
    with torch.cuda.device(dev):
        _host_call(target_logits, draft_logits, draft_tokens, draft_len, temperature, uniforms,
                   uniforms_resample, B, K, V, accepted_len, out_tokens, staging, workspace,
                   _stream_ptr(stream, dev))
    return accepted_len, out_tokens


def _host_call(target_logits, draft_logits, draft_tokens, draft_len, temperature, uniforms,
               uniforms_resample, B, K, V, accepted_len, out_tokens, staging, workspace, stream):
    check("spec_verify_sample_host", lib().spec_verify_sample_host(
        _ptr(target_logits), _ptr(draft_logits), _dtype_code(target_logits), _ptr(draft_tokens),
        _ptr(draft_len), _ptr(temperature), _ptr(uniforms), _ptr(uniforms_resample), B, K, V,
        _ptr(accepted_len), _ptr(out_tokens), staging.tensor.data_ptr(), staging.nbytes,
        workspace.tensor.data_ptr(), workspace.nbytes, stream))


def spec_verify_sample_noalloc(target_logits, draft_logits, draft_tokens, draft_len, temperature,
                               uniforms, uniforms_resample, *, accepted_len, out_tokens,
                               stream=None):
    """The sampler for callers that cannot allocate device memory at the call
    site (plugin hooks handed only their declared tensors, serving loops that
    forbid cudaMalloc after start-up, hosts whose memory another allocator
    owns).  The caller passes preallocated outputs; the scratch is the
    library's own fixed 4 MiB device array (shapes whose workspace exceeds
    it are rejected), shared by every call on the device, so calls that may
    overlap on the GPU must be serialised.  Make the first call on a
    device before any stream capture: it looks up the array's address."""
    B, K, V = _check_inputs(target_logits, draft_logits, draft_tokens, draft_len, temperature,
                            uniforms, uniforms_resample)
    torch = _torch()
    dev = target_logits.device
    for name, t, shape in (("accepted_len", accepted_len, (B,)),
                           ("out_tokens", out_tokens, (B, K + 1))):
        if (t is None or tuple(t.shape) != shape or t.dtype != torch.int32 or t.device != dev
                or not t.is_contiguous()):
            raise ValueError(f"{name} must be a preallocated int32 tensor {shape} on {dev}")
    with torch.cuda.device(dev):   # its scratch array is the current device's
        check("spec_verify_sample_noalloc", lib().spec_verify_sample_noalloc(
            _ptr(target_logits), _ptr(draft_logits), _dtype_code(target_logits),
            _ptr(draft_tokens), _ptr(draft_len), _ptr(temperature), _ptr(uniforms),
            _ptr(uniforms_resample), B, K, V, _ptr(accepted_len), _ptr(out_tokens),
            _stream_ptr(stream, dev)))
    return accepted_len, out_tokens


def _need(name, t, shape, dtype, dev):
    torch = _torch()
    if t is None or tuple(t.shape) != tuple(shape) or t.dtype != dtype or t.device != dev \
            or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {dtype} tensor of shape {tuple(shape)} "
                         f"on {dev}")


def sample_draft(logits, temperature, uniforms, *, workspace=None, tokens=None, row_stats=None,
                 stream=None):
    """The draft-side sampler: one token per row of ``logits`` [R, V]
    (bf16/f32) from softmax(z / T) with ``uniforms`` [R]; the row's argmax
    where T = 0.  Returns tokens [R] int32 (asynchronous)."""
    torch = _torch()
    if logits.dim() != 2:
        raise ValueError("logits must be [R, V]")
    R, V = logits.shape
    dev = logits.device
    _need("logits", logits, (R, V), logits.dtype, dev)
    _need("temperature", temperature, (R,), torch.float32, dev)
    _need("uniforms", uniforms, (R,), torch.float32, dev)
    if tokens is None:
        tokens = torch.empty(R, dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = Workspace(R, 0, V, logits.dtype, dev, stream, kind="sample")
    with torch.cuda.device(dev):
        check("spec_sample_draft", lib().spec_sample_draft(
            _ptr(logits), _dtype_code(logits), _ptr(temperature), _ptr(uniforms), R, V,
            _ptr(tokens), workspace.tensor.data_ptr(), workspace.nbytes, _ptr(row_stats),
            _stream_ptr(stream, dev)))
    return tokens


def spec_verify_sample_onehot(target_logits, draft_tokens, draft_len, temperature, uniforms,
                              uniforms_resample, *, workspace=None, accepted_len=None,
                              out_tokens=None, row_stats=None, stream=None):
    """Verification for a draft that proposes its top token (no draft
    logits: q is the point mass at each drafted token).  Tensors as for
    spec_verify_sample without draft_logits.  Returns (accepted_len [B],
    out_tokens [B, K+1]) int32 (asynchronous)."""
    torch = _torch()
    B, K, V = _check_inputs(target_logits, None, draft_tokens, draft_len, temperature, uniforms,
                            uniforms_resample)
    dev = target_logits.device
    if accepted_len is None:
        accepted_len = torch.empty(B, dtype=torch.int32, device=dev)
    if out_tokens is None:
        out_tokens = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = Workspace(B, K, V, target_logits.dtype, dev, stream)
    with torch.cuda.device(dev):
        check("spec_verify_sample_onehot", lib().spec_verify_sample_onehot(
            _ptr(target_logits), _dtype_code(target_logits), _ptr(draft_tokens), _ptr(draft_len),
            _ptr(temperature), _ptr(uniforms), _ptr(uniforms_resample), B, K, V,
            _ptr(accepted_len), _ptr(out_tokens), workspace.tensor.data_ptr(), workspace.nbytes,
            _ptr(row_stats), _stream_ptr(stream, dev)))
    return accepted_len, out_tokens


def verify_tree_greedy(target_logits, parents, tokens, n_nodes, *, workspace=None,
                       accepted_len=None, out_tokens=None, path_nodes=None, row_stats=None,
                       stream=None):
    """Greedy verification of token trees: ``target_logits`` [B, N, V] (row i
    = the target's logits at node i), ``parents`` [B, N] int32 (-1 at the
    root, else < i), ``tokens`` [B, N] int32, ``n_nodes`` [B] int32.  Returns
    (accepted_len [B], out_tokens [B, N], path_nodes [B, N]) int32."""
    torch = _torch()
    if target_logits.dim() != 3:
        raise ValueError("target_logits must be [B, N, V]")
    B, N, V = target_logits.shape
    dev = target_logits.device
    _need("target_logits", target_logits, (B, N, V), target_logits.dtype, dev)
    _dtype_code(target_logits)
    _need("parents", parents, (B, N), torch.int32, dev)
    _need("tokens", tokens, (B, N), torch.int32, dev)
    _need("n_nodes", n_nodes, (B,), torch.int32, dev)
    if accepted_len is None:
        accepted_len = torch.empty(B, dtype=torch.int32, device=dev)
    if out_tokens is None:
        out_tokens = torch.empty((B, N), dtype=torch.int32, device=dev)
    if path_nodes is None:
        path_nodes = torch.empty((B, N), dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = Workspace(B, N, V, target_logits.dtype, dev, stream, kind="tree")
    with torch.cuda.device(dev):
        check("spec_verify_tree_greedy", lib().spec_verify_tree_greedy(
            _ptr(target_logits), _dtype_code(target_logits), _ptr(parents), _ptr(tokens),
            _ptr(n_nodes), B, N, V, _ptr(accepted_len), _ptr(out_tokens), _ptr(path_nodes),
            workspace.tensor.data_ptr(), workspace.nbytes, _ptr(row_stats),
            _stream_ptr(stream, dev)))
    return accepted_len, out_tokens, path_nodes


def insert_accepted(accepted_len, out_tokens, seq_lens, history, *, next_tokens=None,
                    cu_emitted=None, packed=None, status=None, stream=None):
    """The post-accept insert on the device: appends each request's emitted
    tokens (out_tokens[b, :accepted_len[b] + 1]) to ``history`` [B, L] at
    ``seq_lens`` [B] (both updated in place) and returns (next_tokens [B],
    cu_emitted [B+1], packed [B*(K+1)], status [B]) int32 (asynchronous)."""
    torch = _torch()
    B, K1 = out_tokens.shape
    L = history.shape[1]
    dev = out_tokens.device
    _need("accepted_len", accepted_len, (B,), torch.int32, dev)
    _need("out_tokens", out_tokens, (B, K1), torch.int32, dev)
    _need("seq_lens", seq_lens, (B,), torch.int32, dev)
    _need("history", history, (B, L), torch.int32, dev)
    if next_tokens is None:
        next_tokens = torch.empty(B, dtype=torch.int32, device=dev)
    if cu_emitted is None:
        cu_emitted = torch.empty(B + 1, dtype=torch.int32, device=dev)
    if packed is None:
        packed = torch.full((B * K1,), -1, dtype=torch.int32, device=dev)
    if status is None:
        status = torch.empty(B, dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        check("spec_insert_accepted", lib().spec_insert_accepted(
            _ptr(accepted_len), _ptr(out_tokens), B, K1 - 1, _ptr(seq_lens), _ptr(history), L,
            _ptr(next_tokens), _ptr(cu_emitted), _ptr(packed), _ptr(status),
            _stream_ptr(stream, dev)))
    return next_tokens, cu_emitted, packed, status
