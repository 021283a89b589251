"""The no-allocation entry point, checked against the workspace entry point.

spec_verify_sample_noalloc serves callers that cannot allocate device memory
where they run the sampler (plugin hooks that only receive their declared
tensors, serving loops that forbid cudaMalloc after start-up, hosts whose
device memory another allocator owns).  Its scratch is the library's fixed
device array, so this file runs it twice in a row on the same device and
compares both results with spec_verify_sample on a caller-owned workspace.
It is collected last on purpose: a failure here leaves every other test run.
"""

import numpy as np
import pytest

from speculative_decoding_verify_sample_gb300 import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _device_args(inp):
    from helpers import to_device
    d = to_device(inp, "cuda")
    return (d["target"], d["draft"], d["draft_tokens"], d["draft_len"], d["temperature"],
            d["uniforms"], d["uniforms_resample"])


@pytest.mark.parametrize("seed,B,K,V,dtype", [(7, 24, 4, 50000, "bf16"), (8, 9, 6, 3001, "f32")])
def test_noalloc_matches_workspace_entry_twice(seed, B, K, V, dtype):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import speculative_decoding_verify_sample_gb300 as sv
    sv.build()
    inp = synth.random_case(seed, B, K, V, dtype, temperature=0.9, draft_len="random",
                            greedy_frac=0.3)
    args = _device_args(inp)
    ws = sv.Workspace(B, K, V, dtype, "cuda")
    acc_ref, out_ref = sv.spec_verify_sample(*args, workspace=ws)
    torch.cuda.synchronize()
    acc_ref, out_ref = acc_ref.cpu().numpy(), out_ref.cpu().numpy()
    assert np.all(acc_ref >= 0)
    for _ in range(2):
        acc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
        out = torch.full((B, K + 1), -7, dtype=torch.int32, device="cuda")
        sv.spec_verify_sample_noalloc(*args, accepted_len=acc, out_tokens=out)
        torch.cuda.synchronize()
        # integer outputs of the same kernel on the same inputs: exact
        assert np.array_equal(acc.cpu().numpy(), acc_ref)
        assert np.array_equal(out.cpu().numpy(), out_ref)
