"""Host-side tests of the C ABI that need no GPU.

The library is built with nvcc (cross-compiling for sm_103a works without a
GPU) and loaded with ctypes.  Checked here: every function declared in
include/gqa_decode.h is exported; workspace sizes; the split planner's table;
and that argument validation returns the documented status before any CUDA
call (the fake device addresses below are never dereferenced).
"""
import ctypes
import os
import re

import pytest

from gqa_decode_attention_sm_gb300 import _lib
from gqa_decode_attention_sm_gb300 import build as gbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "gqa_decode.h")

OK, EINVAL, EDEV, EWS, EALIAS, ECUDA = 0, 1, 2, 3, 4, 5
F16, BF16 = 0, 1
KV_F16, KV_BF16, KV_E4M3, KV_I8 = 0, 1, 2, 3


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return _lib.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gqa_[a-z0-9_]+)\s*\(", text)))


def test_header_and_binding_agree():
    assert _declared_functions() == sorted(_lib.EXPORTS)


def test_library_exports_every_declared_function(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="missing"):
        _lib.load(str(tmp_path / "libnothing.so"))


def test_status_strings(lib):
    names = [lib.gqa_status_string(i).decode() for i in range(6)]
    assert names == ["GQA_OK", "GQA_ERR_INVALID_ARGUMENT", "GQA_ERR_UNSUPPORTED_DEVICE",
                     "GQA_ERR_WORKSPACE_TOO_SMALL", "GQA_ERR_ALIASING", "GQA_ERR_CUDA"]


def _ws_expected(B, S):
    if S == 1:
        return 256
    up = lambda x: (x + 255) // 256 * 256  # noqa: E731
    return 256 + up(B * 32 * S * 128 * 4) + 2 * up(B * 32 * S * 4)


@pytest.mark.parametrize("B,C,S", [(1, 64, 1), (1, 1024, 16), (8, 131072, 19), (64, 32768, 3),
                                   (32, 8192, 256), (3, 5, 7)])
def test_workspace_size(lib, B, C, S):
    assert lib.gqa_decode_workspace_size(B, C, S) == _ws_expected(B, S)


@pytest.mark.parametrize("args", [(0, 64, 1), (1, 0, 1), (1, 64, 0), (1, 64, 257), (-1, 64, 2)])
def test_workspace_size_invalid(lib, args):
    assert lib.gqa_decode_workspace_size(*args) == 0


def _plan(lib, B, C, fmt, sms):
    n = ctypes.c_int(-1)
    st = lib.gqa_decode_plan_for(B, C, fmt, sms, ctypes.byref(n))
    return st, n.value


def _chunk(C, S, fmt):
    tile = 128 if fmt == KV_E4M3 else 64
    per = -(-C // S)
    return -(-per // tile) * tile


# (batch, capacity, format, SM count) -> splits: about 8 waves of work items
# (2 resident per SM for 16-bit KV, 3 for 8-bit KV) over the worst case, or,
# when all rows hold at most 16 tiles per resident slot, about sqrt(6 * tiles
# per row), capped at one wave unless the batch has 8 or more rows of 4096
# slots or more (then the balanced schedule takes the grid); whole tiles per
# split (at least two), 1..256.
PLAN_TABLE = [
    ((1, 64, KV_F16, 152), 1),
    ((1, 1024, KV_F16, 152), 8),
    ((32, 8192, KV_F16, 152), 10),
    ((8, 131072, KV_BF16, 152), 38),
    ((64, 32768, KV_E4M3, 152), 8),
    ((1, 1 << 18, KV_BF16, 152), 256),
    ((1, 1 << 22, KV_BF16, 400), 256),
    ((1, 1, KV_F16, 152), 1),
    ((65535, 64, KV_F16, 152), 1),
    ((2, 65536, KV_BF16, 100), 94),
    # latency-bound sizes: about sqrt(6 * tiles per row) splits, one wave at most
    ((1, 4096, KV_BF16, 152), 16),
    ((1, 16384, KV_BF16, 152), 37),
    ((4, 4096, KV_BF16, 152), 8),
    ((1, 8192, KV_E4M3, 152), 16),
    ((8, 2048, KV_BF16, 152), 4),
    ((32, 512, KV_BF16, 152), 1),
    # batches of 8+ rows of 4096+ slots: not capped at one wave
    ((8, 4096, KV_BF16, 152), 16),
    ((16, 4096, KV_E4M3, 152), 11),
]


@pytest.mark.parametrize("args,want", PLAN_TABLE)
def test_plan_table(lib, args, want):
    st, S = _plan(lib, *args)
    assert st == OK and S == want


@pytest.mark.parametrize("B,C,fmt", [(b, c, f) for b in (1, 3, 8, 64) for c in (1, 63, 64, 65, 1000, 131072)
                                     for f in (KV_F16, KV_E4M3)])
def test_plan_invariants(lib, B, C, fmt):
    st, S = _plan(lib, B, C, fmt, 152)
    assert st == OK and 1 <= S <= 256
    chunk = _chunk(C, S, fmt)
    tile = 128 if fmt == KV_E4M3 else 64
    assert chunk % tile == 0 and chunk * S >= C
    splits_eff = -(-C // chunk)
    assert 1 <= splits_eff <= S


def test_noalloc_auto_plan_fits_the_static_scratch(lib):
    # gqa_decode_noalloc lowers an automatic split count whose scratch would
    # not fit its 16 MiB static array.  On GB300's SM count (152; 160 for the
    # full die) that lowering never triggers: the planner keeps
    # batch x splits near the resident CTA count, and the largest automatic
    # scratch over batches 1..65535 and capacities 1..2^30 is about 10 MB.  So
    # the lowering loop is only a guard, and this pins why.
    batches = sorted(set(range(1, 400)) | {456, 512, 1000, 1024, 1025, 4096, 65535})
    caps = [1, 16, 64, 65, 129, 300, 1000, 1024, 4096, 8192, 32768, 131072, 1 << 20, 1 << 30]
    for sms in (152, 160):
        worst = 0
        for fmt in (KV_F16, KV_BF16):
            for B in batches:
                for C in caps:
                    st, S = _plan(lib, B, C, fmt, sms)
                    assert st == OK
                    worst = max(worst, lib.gqa_decode_workspace_size(B, C, S))
        assert worst <= (16 << 20) * 0.7, (sms, worst)


@pytest.mark.parametrize("C,S,fmt,chunk,eff", [(64, 1, KV_F16, 64, 1), (1024, 16, KV_F16, 64, 16),
                                                (1000, 7, KV_F16, 192, 6), (1000, 256, KV_E4M3, 128, 8),
                                                (131072, 19, KV_BF16, 6912, 19), (1, 3, KV_F16, 64, 1)])
def test_split_geometry(lib, C, S, fmt, chunk, eff):
    a, b = ctypes.c_int(0), ctypes.c_int(0)
    assert lib.gqa_decode_split_geometry(C, S, fmt, ctypes.byref(a), ctypes.byref(b)) == OK
    assert (a.value, b.value) == (chunk, eff) == (_chunk(C, S, fmt), -(-C // _chunk(C, S, fmt)))


@pytest.mark.parametrize("B,C,fmt,T,S,launches", [
    (1, 64, KV_F16, 1, 1, 1),            # one split: the split kernel writes the output
    (1, 1024, KV_F16, 1, 8, 1),          # 8 splits, one wave: merged on chip in a cluster
    (1, 1024, KV_F16, 4, 8, 1),          # the same with a 4-token window
    (1, 1024, KV_F16, 1, 16, 2),         # 16 splits: more than a portable cluster holds
    (8, 131072, KV_BF16, 1, 38, 2),      # balanced grid + combine
    (32, 8192, KV_F16, 1, 10, 2),        # ragged workload shape: balanced + combine
    (64, 32768, KV_E4M3, 1, 8, 2),       # 8-bit, balanced at 3 CTAs per SM
    (1, 100, KV_F16, 1, 256, 1),         # 256 splits asked, 2 hold slots: cluster of 2
])
def test_launch_count(lib, B, C, fmt, T, S, launches):
    n = ctypes.c_int(0)
    assert lib.gqa_decode_launch_count_for(B, C, fmt, T, S, 152, ctypes.byref(n)) == OK
    assert n.value == launches


def test_launch_count_rejects_bad_arguments(lib):
    n = ctypes.c_int(0)
    assert lib.gqa_decode_launch_count_for(1, 64, KV_F16, 0, 1, 152, ctypes.byref(n)) == EINVAL
    assert lib.gqa_decode_launch_count_for(1, 64, KV_F16, 5, 1, 152, ctypes.byref(n)) == EINVAL
    assert lib.gqa_decode_launch_count_for(1, 64, KV_F16, 1, 0, 152, ctypes.byref(n)) == EINVAL
    assert lib.gqa_decode_launch_count_for(1, 64, KV_F16, 1, 1, 0, ctypes.byref(n)) == EINVAL
    assert lib.gqa_decode_launch_count_for(1, 64, 9, 1, 1, 152, ctypes.byref(n)) == EINVAL
    assert lib.gqa_decode_launch_count_for(1, 64, KV_F16, 1, 1, 152, None) == EINVAL


def test_plan_rejects_bad_arguments(lib):
    assert _plan(lib, 0, 64, KV_F16, 152)[0] == EINVAL
    assert _plan(lib, 1, 64, 7, 152)[0] == EINVAL
    assert _plan(lib, 1, 64, KV_F16, 0)[0] == EINVAL
    assert lib.gqa_decode_plan_for(1, 64, KV_F16, 152, None) == EINVAL


# Fake, well-aligned device addresses: validation must fail before any use.
Q, KV, LENS, OUT, WS = 0x10000000, 0x20000000, 0x30000000, 0x40000000, 0x50000000


def _prepared(lib, **kw):
    a = dict(q=Q, kv=KV, lens=LENS, out=OUT, B=2, C=64, dtype=F16, q_scale=1.0, S=1, ws=WS,
             ws_bytes=256, stream=None)
    a.update(kw)
    return lib.gqa_decode_prepared(a["q"], a["kv"], a["lens"], a["out"], a["B"], a["C"], a["dtype"],
                                   a["q_scale"], a["S"], a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("kw,want", [
    (dict(q=None), EINVAL), (dict(kv=None), EINVAL), (dict(lens=None), EINVAL),
    (dict(out=None), EINVAL), (dict(ws=None), EINVAL),
    (dict(B=0), EINVAL), (dict(B=70000), EINVAL), (dict(C=0), EINVAL),
    (dict(dtype=2), EINVAL),
    (dict(q_scale=0.0), EINVAL), (dict(q_scale=-1.0), EINVAL), (dict(q_scale=float("inf")), EINVAL),
    (dict(q_scale=float("nan")), EINVAL),
    (dict(S=-1), EINVAL), (dict(S=257), EINVAL),
    (dict(q=Q + 8), EINVAL), (dict(kv=KV + 4), EINVAL), (dict(out=OUT + 2), EINVAL),
    (dict(lens=LENS + 2), EINVAL), (dict(ws=WS + 8), EINVAL),
    (dict(S=4, ws_bytes=256), EWS), (dict(ws_bytes=100), EWS),
    (dict(out=Q), EALIAS), (dict(out=KV + 4096), EALIAS), (dict(out=LENS - 16), EALIAS),
    (dict(ws=OUT + 1024), EALIAS), (dict(ws=KV + 256), EALIAS),
])
def test_prepared_validation(lib, kw, want):
    assert _prepared(lib, **kw) == want
    assert lib.gqa_last_error().decode() != ""


def test_fp8_validation(lib):
    f = lib.gqa_decode_fp8kv
    assert f(Q, KV, LENS, OUT, 2, 64, 1.0, 0.0, 1.0, 1, WS, 256, None) == EINVAL   # k_scale 0
    assert f(Q, KV, LENS, OUT, 2, 64, 1.0, 1.0, -2.0, 1, WS, 256, None) == EINVAL  # v_scale < 0
    assert f(Q, KV, LENS, OUT, 2, 64, 1.0, 1.0, float("inf"), 1, WS, 256, None) == EINVAL
    assert f(Q, KV, LENS, OUT, 2, 64, -1.0, 1.0, 1.0, 1, WS, 256, None) == EINVAL  # q_scale < 0
    assert f(Q, KV, LENS, OUT, 2, 64, 1.0, 1.0, 1.0, 3, WS, 256, None) == EWS


def test_stage_validation(lib):
    s = lib.gqa_decode_split_stage
    # fp16 KV with bf16 q is rejected; e4m3 KV accepts either q dtype
    assert s(Q, BF16, KV, KV_F16, LENS, OUT, 2, 64, 1.0, 1.0, 1.0, 1, WS, 256, None) == EINVAL
    assert s(Q, F16, KV, 9, LENS, OUT, 2, 64, 1.0, 1.0, 1.0, 1, WS, 256, None) == EINVAL
    c = lib.gqa_decode_combine_stage
    assert c(None, OUT, F16, KV_F16, 2, 64, 1.0, 1, WS, 256, None) == EINVAL
    assert c(LENS, OUT, F16, KV_F16, 2, 64, 0.0, 1, WS, 256, None) == EINVAL
    assert c(LENS, OUT, F16, KV_F16, 2, 64, 1.0, 4, WS, 256, None) == EWS
    assert c(LENS, WS + 64, F16, KV_F16, 2, 64, 1.0, 1, WS, 256, None) == EALIAS


def test_int8_validation(lib):
    f = lib.gqa_decode_int8kv
    SC = 0x60000000
    assert f(Q, KV, None, LENS, OUT, 2, 64, F16, 1.0, 1, WS, 256, None) == EINVAL      # no scales
    assert f(Q, KV, SC + 2, LENS, OUT, 2, 64, F16, 1.0, 1, WS, 256, None) == EINVAL    # misaligned
    assert f(Q, KV, SC, LENS, OUT, 2, 60, F16, 1.0, 1, WS, 256, None) == EINVAL        # capacity % 8
    assert f(Q, KV, SC, LENS, OUT, 2, 64, 7, 1.0, 1, WS, 256, None) == EINVAL          # dtype
    assert f(Q, KV, SC, LENS, SC + 64, 2, 64, F16, 1.0, 1, WS, 256, None) == EALIAS    # out on scales
    assert f(Q, KV, SC, LENS, OUT, 2, 64, F16, 1.0, 4, WS, 256, None) == EWS
    # stage 1 alone has no scale argument, so it refuses an int8 cache
    assert lib.gqa_decode_split_stage(Q, F16, KV, KV_I8, LENS, OUT, 2, 64, 1.0, 1.0, 1.0, 1, WS, 256,
                                      None) == EINVAL
    # 8-bit formats share the 128-token tile
    a, b = ctypes.c_int(0), ctypes.c_int(0)
    assert lib.gqa_decode_split_geometry(1000, 256, KV_I8, ctypes.byref(a), ctypes.byref(b)) == OK
    assert (a.value, b.value) == (128, 8)


def test_paged_validation(lib):
    f = lib.gqa_decode_paged
    BT = 0x70000000

    def call(**kw):
        a = dict(q=Q, qd=F16, kv=KV, kvf=KV_F16, sc=None, bt=BT, maxp=4, nump=16, ps=64, lens=LENS, out=OUT,
                 B=2, T=1, S=1, ws=WS, wsb=256)
        a.update(kw)
        return f(a["q"], a["qd"], a["kv"], a["kvf"], a["sc"], a["bt"], a["maxp"], a["nump"], a["ps"],
                 a["lens"], a["out"], a["B"], a["T"], 1.0, 1.0, 1.0, a["S"], a["ws"], a["wsb"], None)

    assert call(bt=None) == EINVAL
    assert call(kvf=KV_I8) == EINVAL                 # int8 without its scale pool
    assert call(kvf=KV_I8, sc=0x60000008) == EINVAL  # scale pool not 16-byte aligned
    assert call(T=0) == EINVAL and call(T=5) == EINVAL
    assert call(ps=48) == EINVAL and call(ps=8) == EINVAL and call(ps=1 << 17) == EINVAL
    assert call(nump=0) == EINVAL and call(maxp=0) == EINVAL
    assert call(maxp=1 << 20, ps=2048) == EINVAL     # capacity above 2^30
    assert call(bt=BT + 2) == EINVAL
    assert call(out=BT) == EALIAS                    # out on the block table
    assert call(S=4) == EWS
    assert call(S=4, T=2, wsb=lib.gqa_decode_workspace_size(2, 256, 4)) == EWS  # the window needs 2 x rows


def test_append_paged_validation(lib):
    f = lib.gqa_append_kv_paged
    P = 0x11000000  # stand-in device addresses (validation fails before any launch)

    def call(**kw):
        a = dict(bt=0x70000000, kvf=KV_F16, sc=None, maxp=4, nump=16, ps=64, ws=None, wsb=0)
        a.update(kw)
        return f(P, P + 0x100000, P + 0x200000, P + 0x300000, P + 0x400000, F16, 0x12000000, 0x12100000, 2,
                 0x13000000, KV, a["kvf"], a["sc"], a["bt"], a["maxp"], a["nump"], a["ps"], 1e-6, 1e6, 1.0,
                 1.0, a["ws"], a["wsb"], None)

    assert call(bt=None) == EINVAL
    assert call(ps=48) == EINVAL and call(ps=8) == EINVAL
    assert call(nump=0) == EINVAL and call(maxp=0) == EINVAL
    assert call(maxp=1 << 20, ps=2048) == EINVAL
    assert call(bt=0x70000002) == EINVAL
    assert call(kvf=KV_I8) == EINVAL  # int8 without its scale pool
    assert call(ws=WS, wsb=8) == EWS


def test_verify_validation(lib):
    f = lib.gqa_decode_verify
    assert f(Q, F16, KV, KV_F16, None, LENS, OUT, 2, 64, 0, 1.0, 1.0, 1.0, 1, WS, 256, None) == EINVAL
    assert f(Q, F16, KV, KV_F16, None, LENS, OUT, 2, 64, 5, 1.0, 1.0, 1.0, 1, WS, 256, None) == EINVAL
    assert f(Q, F16, KV, KV_I8, None, LENS, OUT, 2, 64, 2, 1.0, 1.0, 1.0, 1, WS, 256, None) == EINVAL
    # the workspace is sized for batch * q_len rows
    need = lib.gqa_decode_workspace_size(2 * 3, 64, 4)
    assert f(Q, F16, KV, KV_F16, None, LENS, OUT, 2, 64, 3, 1.0, 1.0, 1.0, 4, WS,
             lib.gqa_decode_workspace_size(2, 64, 4), None) == EWS
    assert need > lib.gqa_decode_workspace_size(2, 64, 4)
    # out spans batch * q_len rows: placing it right after q's first row overlaps
    assert f(Q, F16, KV, KV_F16, None, LENS, Q + 2 * 32 * 128 * 2, 2, 64, 3, 1.0, 1.0, 1.0, 1, WS, 256,
             None) == EALIAS


def test_append_validation(lib):
    f = lib.gqa_append_kv
    QP, KP, VP, WQ, WK, POS, SL, QO, KVC = (0x10000000 + i * 0x1000000 for i in range(9))

    def call(**kw):
        a = dict(qp=QP, kp=KP, vp=VP, wq=WQ, wk=WK, dt=BF16, pos=POS, sl=SL, B=2, qo=QO, kv=KVC,
                 fmt=KV_BF16, sc=None, C=64, eps=1e-6, th=1e6, ks=1.0, vs=1.0, ws=None, wsb=0)
        a.update(kw)
        return f(a["qp"], a["kp"], a["vp"], a["wq"], a["wk"], a["dt"], a["pos"], a["sl"], a["B"], a["qo"],
                 a["kv"], a["fmt"], a["sc"], a["C"], a["eps"], a["th"], a["ks"], a["vs"], a["ws"], a["wsb"],
                 None)

    assert call(qp=None) == EINVAL and call(sl=None) == EINVAL
    assert call(fmt=KV_F16) == EINVAL                 # fp16 cache with bf16 projections
    assert call(fmt=KV_I8) == EINVAL                  # int8 cache without scales
    assert call(eps=-1.0) == EINVAL and call(th=0.0) == EINVAL and call(ks=0.0, fmt=KV_E4M3) == EINVAL
    assert call(ws=WS, wsb=16) == EWS
    assert call(qp=QP + 1) == EINVAL
    assert call(qo=QP) == EALIAS                      # q_out on q_proj
    assert call(kv=KP) == EALIAS                      # cache on k_proj


def test_convenience_validation(lib):
    g = lib.gqa_decode
    assert g(None, KV, LENS, OUT, 1, 64, F16, 1.0, None) == EINVAL
    assert g(Q, KV, LENS, OUT, 1, 64, F16, -0.5, None) == EINVAL
    assert g(Q, KV, LENS, Q, 1, 64, F16, 1.0, None) == EALIAS


def test_status_calls_validate(lib):
    flags = ctypes.c_uint32(0)
    assert lib.gqa_decode_get_status(None, 256, None, ctypes.byref(flags)) == EINVAL
    assert lib.gqa_decode_get_status(WS, 16, None, ctypes.byref(flags)) == EINVAL
    assert lib.gqa_decode_workspace_init(None, 256, None) == EINVAL
    assert lib.gqa_decode_workspace_init(WS, 8, None) == EINVAL
    assert lib.gqa_decode_noalloc_get_status(None, None) == EINVAL


def test_extent_cuts_are_refused_by_the_product_build(lib):
    # the product library carries no range checks: only "no cut" is accepted
    assert lib.gqa_decode_debug_cut_extents(0, 0) == 0
    assert lib.gqa_decode_debug_cut_extents(1, 0) == EINVAL
    assert lib.gqa_decode_debug_cut_extents(0, 4096) == EINVAL
    assert "checked build" in lib.gqa_last_error().decode()


def test_status_flags_agree_with_the_header():
    # every GQA_FLAG_* of the header has the binding's value
    text = open(HEADER).read()
    flags = dict(re.findall(r"#define GQA_FLAG_([A-Z_]+)\s+(0x[0-9a-fA-F]+)u", text))
    from gqa_decode_attention_sm_gb300 import api
    assert flags, "no GQA_FLAG_* in the header"
    for name, value in flags.items():
        assert getattr(api, "FLAG_" + name) == int(value, 16), name
