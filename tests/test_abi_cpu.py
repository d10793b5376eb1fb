"""The C ABI library builds for sm_103a, loads, and exports every entry point that
include/dflash2.h declares. Host-only: no GPU call is made."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from block_drafter_dflash2_gb300 import _build
    import block_drafter_dflash2_gb300 as df2
    _build.build()
    return df2.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "dflash2.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dflash2_[a-z_0-9]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"dflash2_conv", "dflash2_select_topk", "dflash2_viterbi", "dflash2_draft_tail",
            "dflash2_workspace_size", "dflash2_read_device_error", "dflash2_status_string"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} not exported"


def test_status_strings_and_version(lib):
    import block_drafter_dflash2_gb300 as df2
    for code in range(6):
        assert len(df2.status_string(code)) >= 2
    assert df2.version() >= 100


def test_invalid_shapes_rejected_before_any_cuda_call(lib):
    import block_drafter_dflash2_gb300 as df2
    bad = [
        df2.Shape.make(1, 8, 5120 + 32, 1000, 16, 256, 5),   # hidden % 64
        df2.Shape.make(1, 8, 5120, 1000, 17, 256, 5),        # top_k > 16
        df2.Shape.make(1, 8, 5120, 10, 16, 256, 5),          # top_k > vocab
        df2.Shape.make(1, 8, 5120, 1000, 16, 250, 5),        # rank % 16
        df2.Shape.make(1, 33, 5120, 1000, 16, 256, 5),       # block > 32
        df2.Shape.make(0, 8, 5120, 1000, 16, 256, 5),        # batch 0
    ]
    for s in bad:
        assert df2.workspace_size(s) == 0
        st = lib.dflash2_draft_tail(ctypes.byref(s), *([None] * 13), 0, None)
        assert st in (df2.ERR_INVALID_ARGUMENT, df2.ERR_UNSUPPORTED)
    s = df2.Shape.make(1, 8, 5120, 1000, 16, 256, 5, conv_group_size=8)
    assert lib.dflash2_conv(ctypes.byref(s), None, None, None, None, 0, None) == df2.ERR_UNSUPPORTED
    assert lib.dflash2_read_device_error(None, None, None) == df2.ERR_INVALID_ARGUMENT
