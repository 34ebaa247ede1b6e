"""ctypes binding of libgdn_b300.so (argument marshalling only).

Every step of the computation runs in the CUDA library; this module only
checks tensor shapes/dtypes, passes raw device pointers and the current CUDA
stream, and turns status codes into exceptions.  If the library is missing it
raises: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

STATUS = {
    0: "GDN_OK", 1: "GDN_ERR_NULL_PTR", 2: "GDN_ERR_BAD_DIM", 3: "GDN_ERR_UNSUPPORTED",
    4: "GDN_ERR_MISALIGNED", 5: "GDN_ERR_ALLOC", 6: "GDN_ERR_LAUNCH", 7: "GDN_ERR_TIMEOUT",
    8: "GDN_ERR_ALIAS", 9: "GDN_ERR_NO_DEVICE", 10: "GDN_ERR_TOO_LARGE",
    11: "GDN_ERR_RANGE",
}
EXPORTS = (
    "gdn_frame_forward", "gdn_frame_forward_reverse", "gdn_frame_step", "gdn_frame_forward_timed",
    "gdn_frame_forward_host", "gdn_frame_forward_gated", "gdn_frame_step_gated",
    "gdn_workspace_bytes", "gdn_step_workspace_bytes",
    "gdn_status_string", "gdn_sync_status", "gdn_set_wait_limit_ns", "gdn_selftest_wait_timeout",
    "gdn_version", "gdn_frame_step_noalloc", "gdn_set_fused_scan", "gdn_scan_schedule",
    "gdn_set_contract_split", "gdn_frame_forward_fp8", "gdn_frame_step_fp8", "gdn_frame_backward",
    "gdn_set_fused_step", "gdn_set_single_pass", "gdn_forward_schedule", "gdn_debug_last_timeout",
    "gdn_frame_forward_nvfp4", "gdn_frame_step_nvfp4", "gdn_set_host_chunk_frames", "gdn_set_contract_pairs",
    "gdn_frame_forward_save", "gdn_frame_backward_saved",
)


class GDNError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        self.status = STATUS.get(code, f"code {code}")
        super().__init__(f"{what}: {self.status}")


_lib = None


def load(path: str | None = None):
    """Load the library (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _build.LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"CUDA library not built: {p} (run frame_wise_gated_forward_b300.build.build())")
    lib = ctypes.CDLL(p)
    vp, fp, i, st = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p
    lib.gdn_frame_forward.argtypes = [vp, vp, vp, fp, fp, fp, vp, fp, i, i, i, i, i, i, st]
    lib.gdn_frame_forward.restype = ctypes.c_int
    lib.gdn_frame_forward_reverse.argtypes = [vp, vp, vp, fp, fp, fp, vp, fp, i, i, i, i, i, i, st]
    lib.gdn_frame_forward_reverse.restype = ctypes.c_int
    fl = ctypes.c_float
    lib.gdn_frame_forward_gated.argtypes = [vp, vp, vp, fp, fp, fl, fp, vp, fp, i, i, i, i, i, i, st]
    lib.gdn_frame_forward_gated.restype = ctypes.c_int
    lib.gdn_frame_step_gated.argtypes = [vp, vp, vp, fp, fp, fl, fp, vp, fp, i, i, i, i, i, st]
    lib.gdn_frame_step_gated.restype = ctypes.c_int
    lib.gdn_frame_forward_fp8.argtypes = [vp, vp, vp, fl, fl, fl, fp, fp, fp, vp, fp, i, i, i, i, i, i, st]
    lib.gdn_frame_forward_fp8.restype = ctypes.c_int
    lib.gdn_frame_step_fp8.argtypes = [vp, vp, vp, fl, fl, fl, fp, fp, fp, vp, fp, i, i, i, i, i, st]
    lib.gdn_frame_step_fp8.restype = ctypes.c_int
    lib.gdn_frame_forward_nvfp4.argtypes = [vp, vp, vp, vp, vp, vp, fl, fl, fl, fp, fp, fp, vp, fp,
                                            i, i, i, i, i, i, st]
    lib.gdn_frame_forward_nvfp4.restype = ctypes.c_int
    lib.gdn_frame_step_nvfp4.argtypes = [vp, vp, vp, vp, vp, vp, fl, fl, fl, fp, fp, fp, vp, fp, i, i, i, i, i, st]
    lib.gdn_frame_step_nvfp4.restype = ctypes.c_int
    lib.gdn_frame_backward.argtypes = [vp, vp, vp, fp, fp, fp, vp, fp, vp, vp, vp, fp, fp, fp,
                                       i, i, i, i, i, i, st]
    lib.gdn_frame_backward.restype = ctypes.c_int
    lib.gdn_frame_backward_saved.argtypes = [vp, vp, vp, fp, fp, fp, vp, vp, vp, fp, vp, vp, vp, fp, fp, fp,
                                             i, i, i, i, i, i, st]
    lib.gdn_frame_backward_saved.restype = ctypes.c_int
    lib.gdn_frame_forward_save.argtypes = [vp, vp, vp, fp, fp, fp, vp, fp, vp, vp, i, i, i, i, i, i, st]
    lib.gdn_frame_forward_save.restype = ctypes.c_int
    lib.gdn_frame_step.argtypes = [vp, vp, vp, fp, fp, fp, vp, fp, i, i, i, i, i, st]
    lib.gdn_frame_step.restype = ctypes.c_int
    lib.gdn_frame_forward_timed.argtypes = [vp, vp, vp, fp, fp, fp, vp, fp, i, i, i, i, i, i, st,
                                            ctypes.POINTER(ctypes.c_void_p)]
    lib.gdn_frame_forward_timed.restype = ctypes.c_int
    lib.gdn_frame_forward_host.argtypes = [vp, vp, vp, fp, fp, fp, vp, fp, i, i, i, i, i, i, st]
    lib.gdn_frame_forward_host.restype = ctypes.c_int
    lib.gdn_workspace_bytes.argtypes = [i] * 6
    lib.gdn_workspace_bytes.restype = ctypes.c_size_t
    lib.gdn_step_workspace_bytes.argtypes = [i] * 5
    lib.gdn_step_workspace_bytes.restype = ctypes.c_size_t
    lib.gdn_status_string.argtypes = [ctypes.c_int]
    lib.gdn_status_string.restype = ctypes.c_char_p
    lib.gdn_sync_status.argtypes = [st]
    lib.gdn_sync_status.restype = ctypes.c_int
    lib.gdn_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
    lib.gdn_set_wait_limit_ns.restype = None
    lib.gdn_selftest_wait_timeout.argtypes = [ctypes.c_ulonglong, st]
    lib.gdn_selftest_wait_timeout.restype = ctypes.c_int
    lib.gdn_frame_step_noalloc.argtypes = [vp, vp, vp, fp, fp, fp, vp, fp, i, i, i, i, i, st]
    lib.gdn_frame_step_noalloc.restype = ctypes.c_int
    lib.gdn_set_fused_scan.argtypes = [ctypes.c_int]
    lib.gdn_set_fused_scan.restype = None
    lib.gdn_set_fused_step.argtypes = [ctypes.c_int]
    lib.gdn_set_fused_step.restype = None
    lib.gdn_set_contract_split.argtypes = [ctypes.c_int]
    lib.gdn_set_contract_split.restype = None
    lib.gdn_set_single_pass.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int]
    lib.gdn_set_single_pass.restype = None
    lib.gdn_forward_schedule.argtypes = [i] * 6
    lib.gdn_forward_schedule.restype = ctypes.c_int
    lib.gdn_scan_schedule.argtypes = [i, i, i]
    lib.gdn_scan_schedule.restype = ctypes.c_int
    lib.gdn_debug_last_timeout.argtypes = [ctypes.POINTER(ctypes.c_int)]
    lib.gdn_debug_last_timeout.restype = ctypes.c_int
    lib.gdn_set_contract_pairs.argtypes = [ctypes.c_int]
    lib.gdn_set_contract_pairs.restype = None
    lib.gdn_set_host_chunk_frames.argtypes = [ctypes.c_int]
    lib.gdn_set_host_chunk_frames.restype = None
    lib.gdn_version.argtypes = []
    lib.gdn_version.restype = ctypes.c_char_p
    if path is None:
        _lib = lib
    return lib


def check(code: int, what: str) -> None:
    if code != 0:
        raise GDNError(code, what)
