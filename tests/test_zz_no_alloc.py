"""The no-allocation entry point (gqa_decode_noalloc), called through the C ABI.

Some callers cannot allocate device memory at call time (a runtime with a
fixed memory budget or its own allocator, a plugin handed only existing
buffers).  gqa_decode_noalloc serves them with a static device scratch array
instead of a caller or stream-ordered workspace.  This test checks that its
output matches the prepared entry point (gqa_decode_prepared, with a
workspace from the caller) within the parity bar the other tests use, on
two calls in a row with different inputs and then the first input again (the
shared scratch keeps the previous call's contents), and that a split count
whose scratch exceeds the array is refused.

The file is named so that pytest collects it last.  It builds what it needs and
passes in a fresh process as well as after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import gqa_decode_attention_sm_gb300 as gq
from gqa_decode_attention_sm_gb300 import _lib, inputs
from helpers import tolerance_ok

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
STATIC_BYTES = 16 << 20


@pytest.fixture(scope="module")
def lib():
    from gqa_decode_attention_sm_gb300 import build as gbuild
    gbuild.build()
    return _lib.load()


def _noalloc(lib, t, out, num_splits=0):
    w = t["workload"]
    stream = torch.cuda.current_stream(DEV).cuda_stream
    dtype = 0 if w.q_dtype == "f16" else 1
    return lib.gqa_decode_noalloc(t["q"].data_ptr(), t["kv"].data_ptr(), t["lens"].data_ptr(),
                                  out.data_ptr(), w.batch, w.capacity, dtype, float(t["q_scale"]),
                                  num_splits, stream)


def _prepared(t):
    out = torch.empty_like(t["q"])
    p = gq.prepare({"Q": t["q"], "KV": t["kv"], "O": out, "sequence_lengths": t["lens"]},
                   q_scale=t["q_scale"])
    gq.launch(p)
    torch.cuda.synchronize(DEV)
    return out


def _rows(x):
    return x.float().cpu().numpy().reshape(-1, 128)


def test_noalloc_matches_prepared_on_consecutive_calls(lib):
    a = inputs.make(inputs.WORKLOADS[3], DEV)                      # fp16, ragged, NaN tails
    b = inputs.make(inputs.custom(4, 20000, 5000, 20000, kv_dtype="bf16"), DEV)
    refs = {"a": _prepared(a), "b": _prepared(b)}
    for name, t in (("a", a), ("b", b), ("a", a)):
        out = torch.full_like(t["q"], float("nan"))
        st = _noalloc(lib, t, out)
        assert st == 0, lib.gqa_last_error().decode()
        torch.cuda.synchronize(DEV)
        ok, err, _ = tolerance_ok(_rows(out), _rows(refs[name]))
        assert ok, f"call on input {name}: max |noalloc - prepared| {err:.3e}"


def test_noalloc_refuses_scratch_beyond_the_static_array(lib):
    t = inputs.make(inputs.custom(64, 4096, 4096), DEV)
    out = torch.empty_like(t["q"])
    need = lib.gqa_decode_workspace_size(64, 4096, 256)
    assert need > STATIC_BYTES
    assert _noalloc(lib, t, out, num_splits=256) == 3  # GQA_ERR_WORKSPACE_TOO_SMALL
    assert "static scratch" in lib.gqa_last_error().decode()
    # the automatic split count fits itself to the array and still matches
    assert _noalloc(lib, t, out, num_splits=0) == 0
    torch.cuda.synchronize(DEV)
    ok, err, _ = tolerance_ok(_rows(out), _rows(_prepared(t)))
    assert ok, f"auto splits: max |noalloc - prepared| {err:.3e}"
