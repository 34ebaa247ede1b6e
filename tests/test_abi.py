"""CPU checks of the C-ABI library: it builds, loads, exports every symbol the
header declares, and rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest
import torch

from frame_wise_gated_forward_b300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_functions()
    for required in ("gdn_frame_forward", "gdn_frame_step", "gdn_workspace_bytes",
                     "gdn_status_string", "gdn_sync_status"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in gdn.h but not exported"
    assert set(declared_functions()) <= set(_lib.EXPORTS)


def test_status_strings(lib):
    for code, name in _lib.STATUS.items():
        assert lib.gdn_status_string(code).decode().startswith(name)


def test_workspace_bytes(lib):
    # A bf16 + U fp32 + per-frame states bf16 for 121*16 items of 128x128,
    # plus one ready count and one split counter per item.  At N = 880 (14
    # chunks of 64 tokens per item) the automatic plan splits nothing.
    items = 121 * 16
    want = items * 128 * 128 * (2 + 4 + 2) + items * 8
    got = lib.gdn_workspace_bytes(1, 16, 121, 880, 128, 128)
    assert want <= got <= want + 4 * 256
    assert lib.gdn_step_workspace_bytes(1, 16, 880, 128, 128) == lib.gdn_workspace_bytes(1, 16, 1, 880, 128, 128)
    # N = 8800 (138 chunks): 1936 = 13*148 + 12 items, the last 12 split into
    # min(138, 148 // 12) = 12 token ranges with fp32 partial sums (no GPU
    # here, so the library plans for 148 SMs)
    partial = 12 * 12 * (128 * 128 + 128 * 128) * 4
    want = items * 128 * 128 * 8 + items * 8 + partial
    assert want <= lib.gdn_workspace_bytes(1, 16, 121, 8800, 128, 128) <= want + 4 * 256
    # the one-frame step of 16 heads at N = 8800: 148 // 16 = 9 ranges per head
    want = 16 * 128 * 128 * 8 + 16 * 8 + 16 * 9 * 2 * 128 * 128 * 4
    assert want <= lib.gdn_step_workspace_bytes(1, 16, 8800, 128, 128) <= want + 4 * 256
    assert lib.gdn_workspace_bytes(0, 16, 121, 880, 128, 128) == 0
    assert lib.gdn_workspace_bytes(1, 16, 121, 880, 96 + 8, 128) == 0


FAKE = 1 << 20  # never dereferenced: validation rejects before any CUDA call


def call_forward(lib, q=FAKE, k=FAKE * 3, v=FAKE * 5, alpha=FAKE * 7, beta=FAKE * 9,
                 s_in=None, out=FAKE * 11, s_out=None, B=1, H=2, F=3, N=16, dk=32, dv=32):
    # spread the fake buffers 1 MiB apart: far larger than these tiny tensors
    return lib.gdn_frame_forward(q, k, v, alpha, beta, s_in, out, s_out, B, H, F, N, dk, dv, None)


def test_validation_null(lib):
    assert call_forward(lib, q=None) == 1
    assert call_forward(lib, out=None) == 1
    assert call_forward(lib, beta=None) == 1


def test_validation_dims(lib):
    assert call_forward(lib, B=0) == 2
    assert call_forward(lib, N=0) == 2
    assert call_forward(lib, F=-1) == 2
    assert call_forward(lib, dk=24) == 3
    assert call_forward(lib, dv=144) == 3
    assert call_forward(lib, dk=8) == 3
    assert call_forward(lib, B=4096, F=4096, N=4096, H=16, dk=128, dv=128) == 2


def test_validation_alignment(lib):
    assert call_forward(lib, q=FAKE + 8) == 4
    assert call_forward(lib, out=FAKE * 11 + 2) == 4
    assert call_forward(lib, alpha=FAKE * 7 + 2) == 4


def test_validation_alias(lib):
    assert call_forward(lib, out=FAKE) == 8            # out == q
    assert call_forward(lib, out=FAKE * 5 + 64) == 8   # out inside v
    assert call_forward(lib, s_in=FAKE * 13, s_out=FAKE * 13 + 16) == 8  # partial overlap


@pytest.mark.skipif(torch.cuda.is_available(), reason="exercises the no-device path")
def test_valid_arguments_without_gpu_report_no_device(lib):
    assert call_forward(lib) == 9
    assert call_forward(lib, s_in=FAKE * 13, s_out=FAKE * 13) == 9  # in-place state is allowed
    assert lib.gdn_frame_step(FAKE, FAKE * 3, FAKE * 5, FAKE * 7, FAKE * 9, None, FAKE * 11, None,
                              1, 2, 16, 32, 32, None) == 9


def test_product_path_has_no_fallback(tmp_path):
    with pytest.raises(RuntimeError, match="not built"):
        _lib.load(str(tmp_path / "missing.so"))
