"""The no-allocation entry point (gqa_decode_noalloc), called through the C ABI.

Some callers cannot allocate device memory at call time: a runtime with a
fixed memory budget or its own allocator, or a plugin handed only existing
buffers.  gqa_decode_noalloc serves them with a static device scratch array
instead of a workspace from the caller or the stream-ordered allocator.

Checked here, on two calls in a row with different inputs and then the first
input again (the shared scratch keeps the previous call's contents):
* the output matches the FP64 oracle at the parity bar the other tests use;
* it is bit for bit the output of the prepared entry (gqa_decode_prepared,
  with a workspace from the caller) at the same split count: both run the
  same kernels on the same plan;
* neither torch's memory pool nor the device's free memory changes across
  the calls (nothing is allocated);
* the status word of the static scratch is read, and cleared, by
  gqa_decode_noalloc_get_status: a clamped length is reported there and the
  flags of in-contract calls stay 0;
* a split count whose scratch exceeds the array is refused.

The file is named so that pytest collects it last.  It builds what it needs and
passes in a fresh process as well as after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import gqa_decode_attention_sm_gb300 as gq
from gqa_decode_attention_sm_gb300 import _lib, api, inputs
from helpers import bits_of, tolerance_ok

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
STATIC_BYTES = 16 << 20
FMT = {"f16": oracle.F16, "bf16": oracle.BF16}


@pytest.fixture(scope="module")
def lib():
    from gqa_decode_attention_sm_gb300 import build as gbuild
    gbuild.build()
    oracle.build()
    return _lib.load()


def _noalloc(lib, t, out, num_splits=0):
    w = t["workload"]
    stream = torch.cuda.current_stream(DEV).cuda_stream
    dtype = 0 if w.q_dtype == "f16" else 1
    return lib.gqa_decode_noalloc(t["q"].data_ptr(), t["kv"].data_ptr(), t["lens"].data_ptr(),
                                  out.data_ptr(), w.batch, w.capacity, dtype, float(t["q_scale"]),
                                  num_splits, stream)


def _status(lib):
    flags = ctypes.c_uint32(0xFFFFFFFF)
    st = lib.gqa_decode_noalloc_get_status(torch.cuda.current_stream(DEV).cuda_stream, ctypes.byref(flags))
    assert st == 0, lib.gqa_last_error().decode()
    return flags.value


def _prepared(t, num_splits=None):
    out = torch.empty_like(t["q"])
    p = gq.prepare({"Q": t["q"], "KV": t["kv"], "O": out, "sequence_lengths": t["lens"]},
                   q_scale=t["q_scale"], num_splits=num_splits)
    gq.launch(p)
    torch.cuda.synchronize(DEV)
    return out, p.num_splits


def _oracle(t):
    w = t["workload"]
    ref, _ = oracle.gqa_decode(bits_of(t["q"]), FMT[w.q_dtype], bits_of(t["kv"]), FMT[w.kv_dtype],
                               t["lens"].cpu().numpy(), q_scale=t["q_scale"])
    return ref


def _rows(x):
    return x.float().cpu().numpy().reshape(-1, 128)


def _bits_equal(x, y):
    return torch.equal(x.view(torch.int16), y.view(torch.int16))


def test_noalloc_matches_oracle_and_prepared_on_consecutive_calls(lib):
    a = inputs.make(inputs.WORKLOADS[3], DEV)                      # fp16, ragged, NaN tails
    b = inputs.make(inputs.custom(4, 20000, 5000, 20000, kv_dtype="bf16"), DEV)
    cases = {"a": a, "b": b}
    refs = {k: _oracle(t) for k, t in cases.items()}
    prepared = {k: _prepared(t) for k, t in cases.items()}        # the automatic plan of both entries
    outs = [torch.full_like(cases[k]["q"], float("nan")) for k in ("a", "b", "a")]
    torch.cuda.synchronize(DEV)
    pool0, free0 = torch.cuda.memory_allocated(DEV), torch.cuda.mem_get_info(DEV)[0]
    for name, out in zip(("a", "b", "a"), outs):
        st = _noalloc(lib, cases[name], out)
        assert st == 0, lib.gqa_last_error().decode()
        torch.cuda.synchronize(DEV)
        assert torch.cuda.memory_allocated(DEV) == pool0
        assert torch.cuda.mem_get_info(DEV)[0] == free0, "device memory was allocated"
        ok, err, _ = tolerance_ok(_rows(out), refs[name])
        assert ok, f"call on input {name}: max |noalloc - oracle| {err:.3e}"
        ref_out, S = prepared[name]
        assert S > 1  # the scratch's partials and the combine are exercised
        assert _bits_equal(out, ref_out), f"call on input {name}: not bitwise the prepared output (splits {S})"
    assert _status(lib) == 0  # in-contract calls raise no flag


def test_noalloc_status_word_reports_clamped_lengths(lib):
    w = inputs.custom(3, 1024, 1024)
    t = inputs.make(w, DEV, lens=[0, 1024 + 5, 700])             # two out-of-contract lengths
    out = torch.empty_like(t["q"])
    _status(lib)                                                   # start from a clear word
    assert _noalloc(lib, t, out) == 0
    assert _status(lib) & api.FLAG_LENGTH_CLAMPED
    assert _status(lib) == 0                                       # read and cleared
    # flags accumulate over calls until read: a clamped call, then a clean one
    good = inputs.make(w, DEV, lens=[5, 1024, 700])
    assert _noalloc(lib, t, out) == 0
    assert _noalloc(lib, good, out) == 0
    assert _status(lib) == api.FLAG_LENGTH_CLAMPED
    torch.cuda.synchronize(DEV)
    ref = _oracle(good)
    ok, err, _ = tolerance_ok(_rows(out), ref)
    assert ok, f"after a clamped call: max |noalloc - oracle| {err:.3e}"


def test_noalloc_refuses_scratch_beyond_the_static_array(lib):
    t = inputs.make(inputs.custom(64, 4096, 4096), DEV)
    out = torch.empty_like(t["q"])
    need = lib.gqa_decode_workspace_size(64, 4096, 256)
    assert need > STATIC_BYTES
    assert _noalloc(lib, t, out, num_splits=256) == 3  # GQA_ERR_WORKSPACE_TOO_SMALL
    assert "static scratch" in lib.gqa_last_error().decode()
    # an explicit count that fits, and the automatic count: bitwise the prepared entry's
    for S in (8, 0):  # 8 splits: 8.5 MB of scratch
        assert _noalloc(lib, t, out, num_splits=S) == 0
        torch.cuda.synchronize(DEV)
        ref_out, S_used = _prepared(t, num_splits=S or None)
        assert _bits_equal(out, ref_out), f"splits {S_used}: not bitwise the prepared output"
    ok, err, _ = tolerance_ok(_rows(out), _oracle(t))
    assert ok, f"auto splits: max |noalloc - oracle| {err:.3e}"
    assert np.isfinite(_rows(out)).all()
