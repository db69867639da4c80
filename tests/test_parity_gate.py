"""The GPU parity tests can fail where they must (CPU only, no GPU).

Two sensitivity pins, each planting a fault in the oracle's output (never in
the CUDA path) and showing the GPU test's bar rejects it.

1. The long-context gate.

At long context the decode outputs are small: an average of ~131072 V rows
has an RMS near 4.6e-3, so the absolute 3e-3 bar of the element-wise parity
test is most of the signal.  A kernel that silently dropped one split of the
sequence would move every output by roughly RMS / sqrt(splits) and could still
pass that bar.  The GPU tests on long contexts therefore also require
max |gpu - oracle| <= 0.05 * RMS(oracle) (``helpers.rms_gate_ok``).

This test shows, with the oracle alone, that the second gate rejects exactly
that fault while the first does not: batch row 0 of the bf16 8 x 131072
workload (drawn as the benchmark draws it), KV head 0, is decoded in full and
again with one split's worth of tokens removed (3456 tokens: the pieces the
balanced schedule cuts each of its 8 rows into on 304 resident CTAs, and the
chunk of the 38-split plan).  The faulty output is rounded to bf16 as a
kernel's would be.  A correctly rounded output passes both gates.
"""
import numpy as np
import pytest

import oracle
from gqa_decode_attention_sm_gb300 import inputs
from helpers import RMS_GATE, bits_of, rms_gate_ok, tolerance_ok

SPLIT_TOKENS = 3456  # 54 tiles of 64 tokens: 131072 / 38 rounded up to whole tiles


@pytest.fixture(scope="module")
def row0():
    oracle.build()
    t = inputs.make_row(inputs.WORKLOADS[4], 0)
    q = bits_of(t["q"])                      # [1, 32, 128]
    kv = bits_of(t["kv"])                    # [1, 2, 8, 131072, 128]
    L = int(t["lens"][0])
    # only KV head 0 is read for query heads 0..3: keep that head, zero the rest
    kv0 = np.zeros_like(kv)
    kv0[0, :, 0] = kv[0, :, 0]
    del kv, t
    full, full_bits = oracle.gqa_decode(q, oracle.BF16, kv0, oracle.BF16, np.array([L], np.int32),
                                        rows=range(4))
    return q, kv0, L, full, full_bits


def _without(kv0, L, s):
    """The same row with tokens [s * SPLIT_TOKENS, (s + 1) * SPLIT_TOKENS) cut out
    (the later ones moved down), and the shorter length."""
    a, b = s * SPLIT_TOKENS, min(L, (s + 1) * SPLIT_TOKENS)
    cut = kv0.copy()
    cut[0, :, 0, a:L - (b - a)] = kv0[0, :, 0, b:L]
    return cut, L - (b - a)


def test_correctly_rounded_output_passes_both_gates(row0):
    _, _, _, full, full_bits = row0
    got = oracle.decode(full_bits, oracle.BF16)
    ok, _, _ = tolerance_ok(got, full)
    assert ok
    gate_ok, ratio = rms_gate_ok(got, full)
    assert gate_ok, f"bf16 rounding alone gives max error / RMS {ratio:.3e}"
    assert ratio < RMS_GATE / 3  # leaves room for the kernels' own FP32 / 16-bit-weight error


@pytest.mark.parametrize("s", [0, 17, 37])
def test_a_dropped_split_passes_the_absolute_bar_but_fails_the_rms_gate(row0, s):
    q, kv0, L, full, _ = row0
    cut, L2 = _without(kv0, L, s)
    _, dropped_bits = oracle.gqa_decode(q, oracle.BF16, cut, oracle.BF16, np.array([L2], np.int32),
                                        rows=range(4))
    got = oracle.decode(dropped_bits, oracle.BF16)
    rms = float(np.sqrt(np.mean(full ** 2)))
    assert 2e-3 < rms < 8e-3  # the long-context regime the gate is for
    ok, err, _ = tolerance_ok(got, full)
    assert ok, f"split {s}: the absolute bar alone already catches it (max err {err:.3e})"
    gate_ok, ratio = rms_gate_ok(got, full)
    assert not gate_ok, f"split {s}: max error / RMS {ratio:.3e} is inside the gate"


# The GPU test of 8-bit caches with a bf16 q of any magnitude
# (test_8bit_cache_takes_a_bf16_q_of_any_magnitude) can fail: a kernel that
# converted q to f16 directly (saturating at 65504, rounding below 6.1e-5 to
# the f16 subnormal grid) is off by far more than the bar on every one of its
# cases.  The same inputs, the oracle on that converted q against the oracle
# on the bf16 q, the faulty output rounded to bf16 as a kernel's would be.
@pytest.mark.parametrize("kv_dtype", ["e4m3", "i8"])
@pytest.mark.parametrize("T", [1, 3])
@pytest.mark.parametrize("case", ["huge", "tiny", "mixed"])
def test_a_saturating_q_conversion_fails_the_q_range_test(kv_dtype, T, case):
    import torch
    oracle.build()
    w = inputs.custom(4, 704, 1, kv_dtype=kv_dtype, kv_std=2.0 if kv_dtype == "e4m3" else 1.0, nan_tail=True,
                      q_len=T)
    t = inputs.make(w, "cpu", lens=[T, 129, 500, 700])
    g = torch.Generator()
    g.manual_seed(7)
    q = torch.randn(t["q"].shape, generator=g, dtype=torch.float32)
    q_scale = 1.0
    if case == "huge":
        q *= 1e6
    elif case == "tiny":
        q *= 1e-7
        q_scale = 2e7
    else:
        q *= (10.0 ** torch.linspace(-7, 6, 32)).view(32, 1)
        q[..., 0] *= 1e3
    qb = q.to(torch.bfloat16)
    fmt = oracle.E4M3 if kv_dtype == "e4m3" else oracle.I8
    kw = dict(q_scale=q_scale, k_scale=t["k_scale"], v_scale=t["v_scale"])
    if kv_dtype == "i8":
        kw["kv_scales"] = bits_of(t["kv_scales"])
    lens = t["lens"].numpy()
    ref, _ = oracle.gqa_decode(bits_of(qb), oracle.BF16, bits_of(t["kv"]), fmt, lens, **kw)
    q16 = qb.float().clamp(-65504, 65504).to(torch.float16)
    _, faulty_bits = oracle.gqa_decode(bits_of(q16), oracle.F16, bits_of(t["kv"]), fmt, lens,
                                       out_fmt=oracle.BF16, **kw)
    ok, err, _ = tolerance_ok(oracle.decode(faulty_bits, oracle.BF16), ref)
    assert not ok, f"the saturating conversion passes the bar (max err {err:.3e})"
