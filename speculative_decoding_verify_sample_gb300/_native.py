"""ctypes binding of libspecverify (the C ABI declared in include/specverify.h).

Argument marshalling only: every step of the sampler runs in the CUDA
library.  There is no CPU fallback; if the library is missing the calls raise.
"""

from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB_PATH

SPECV_F32 = 0
SPECV_BF16 = 1

STATUS_NAMES = {0: "SPECV_OK", 1: "SPECV_ERR_INVALID_ARG", 2: "SPECV_ERR_UNSUPPORTED",
                3: "SPECV_ERR_WORKSPACE", 4: "SPECV_ERR_CUDA", 5: "SPECV_ERR_BAD_INPUT"}

DEV_BAD_DRAFT_LEN = 0x01
DEV_BAD_TOKEN = 0x02
DEV_BAD_TEMPERATURE = 0x04
DEV_BAD_UNIFORM = 0x08
DEV_BAD_ROW = 0x10
DEV_NO_DRAFT = 0x20
DEV_TIMEOUT = 0x40
DEV_BAD_TREE = 0x80

# exported function -> (restype, argtypes)
_vp = ctypes.c_void_p
_i = ctypes.c_int
_sz = ctypes.c_size_t
_VERIFY_ARGS = [_vp, _vp, _i, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _vp, _vp, _vp, _sz]
SIGNATURES = {
    "specv_version": (_i, []),
    "specv_max_vocab": (_i, [_i]),
    "specv_status_string": (ctypes.c_char_p, [_i]),
    "specv_workspace_bytes": (_sz, [_i, _i, _i, _i]),
    "specv_workspace_init": (_i, [_vp, _sz, _vp]),
    "spec_verify_sample": (_i, _VERIFY_ARGS + [_vp]),
    "spec_verify_sample_debug": (_i, _VERIFY_ARGS + [_vp, _vp]),
    "specv_read_device_status": (_i, [_vp, _sz, _vp, _vp]),
    "specv_host_staging_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "spec_verify_sample_host": (_i, [_vp, _vp, _i, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _vp, _vp,
                                     _vp, _sz, _vp, _sz, _vp]),
    "specv_launch_plan": (_i, [_i, _i, _i, _i, _i, _vp]),
    "spec_verify_sample_noalloc": (_i, [_vp, _vp, _i, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _vp, _vp,
                                        _vp]),
    "specv_sample_workspace_bytes": (_sz, [_i, _i, _i]),
    "spec_sample_draft": (_i, [_vp, _i, _vp, _vp, _i, _i, _vp, _vp, _sz, _vp, _vp]),
    "spec_verify_sample_onehot": (_i, [_vp, _i, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _vp, _vp,
                                       _vp, _sz, _vp, _vp]),
    "specv_tree_workspace_bytes": (_sz, [_i, _i, _i, _i]),
    "spec_verify_tree_greedy": (_i, [_vp, _i, _vp, _vp, _vp, _i, _i, _i, _vp, _vp, _vp, _vp, _sz,
                                     _vp, _vp]),
    "spec_insert_accepted": (_i, [_vp, _vp, _i, _i, _vp, _vp, _i, _vp, _vp, _vp, _vp, _vp]),
}

NOALLOC_SCRATCH_BYTES = 4 << 20

_lock = threading.Lock()
_lib = None


class SpecVerifyError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(status, status)}")


def lib():
    """The loaded library.  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is not built; run speculative_decoding_verify_sample_gb300.build() "
                    "(there is no CPU fallback)")
            try:  # let torch load its CUDA runtime first, when present
                import torch  # noqa: F401
            except ImportError:
                pass
            handle = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
    return _lib


def check(fn: str, status: int):
    if status != 0:
        raise SpecVerifyError(fn, status)
