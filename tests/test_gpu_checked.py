"""The kernels' own range checks, in place of a memory checker (GPU).

No memory checker runs on the GPUs these tests use, so the library is built a
second time with every global-memory access of the split, combine and append
kernels range-checked (`build.build_checked()`, -DGQA_CHECKED).  An access
outside its buffer would set GQA_FLAG_BOUNDS in the status word and be
redirected inside the buffer, so nothing can fault.  The cases below take
every launch path through the checked library: the balanced grid and the
one-piece grid, the combine kernel and the cluster merge, every KV format,
verify windows, paged caches, the int8 tail of scales loaded one by one,
out-of-contract lengths and page ids (clamped on purpose), the staged calls,
the append step and the no-allocation entry.  Each must match the oracle
and leave GQA_FLAG_BOUNDS clear.
"""
import ctypes
import zlib

import numpy as np
import pytest
import torch

import oracle
import gqa_decode_attention_sm_gb300 as gq
from gqa_decode_attention_sm_gb300 import _lib, api, inputs
from helpers import bits_of, tolerance_ok

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
FMT = {"f16": oracle.F16, "bf16": oracle.BF16, "e4m3": oracle.E4M3, "i8": oracle.I8}
FLAG_BOUNDS = api.FLAG_BOUNDS


@pytest.fixture(scope="module", autouse=True)
def checked_library():
    """The checked library in place of the product one for this module."""
    from gqa_decode_attention_sm_gb300 import build as gbuild
    path = gbuild.build_checked()
    oracle.build()
    saved = _lib._lib
    _lib._lib = _lib.load(path)
    yield _lib._lib
    _lib._lib = saved


def _oracle(t, lens=None):
    w = t["workload"]
    lens = t["lens"].cpu().numpy() if lens is None else np.asarray(lens, np.int32)
    args = dict(q_scale=t["q_scale"], k_scale=t["k_scale"], v_scale=t["v_scale"])
    if t.get("kv_scales") is not None:
        args["kv_scales"] = bits_of(t["kv_scales"])
    out, _ = oracle.gqa_decode(bits_of(t["q"]), FMT[w.q_dtype], bits_of(t["kv"]), FMT[w.kv_dtype], lens, **args)
    return out


def _rows(x):
    return x.float().cpu().numpy().reshape(-1, 128)


def _check(flags, what):
    assert not flags & FLAG_BOUNDS, f"{what}: a range check failed (flags {flags:#x})"


def test_uses_the_checked_library(checked_library):
    assert _lib.load() is checked_library


@pytest.mark.parametrize("index", [1, 2, 3])
def test_workloads(index):
    t = inputs.make(inputs.WORKLOADS[index], DEV)
    p = gq.prepare({"Q": t["q"], "KV": t["kv"], "O": torch.empty_like(t["q"]), "sequence_lengths": t["lens"]})
    gq.launch(p)
    _check(gq.get_status(p), f"workload {index}")
    ok, err, _ = tolerance_ok(_rows(p.out), _oracle(t))
    assert ok, f"workload {index}: max err {err:.3e}"


def _window(kv_dtype, B, C, T, lens, S, paged=False, page=64):
    w = inputs.custom(B, C, 1, kv_dtype=kv_dtype, kv_std=2.0 if kv_dtype == "e4m3" else 1.0, nan_tail=True,
                      q_len=T)
    t = inputs.make(w, DEV, lens=lens)
    fp8 = dict(k_scale=t["k_scale"], v_scale=t["v_scale"]) if kv_dtype == "e4m3" else {}
    q4 = t["q"] if T > 1 else t["q"][:, None].contiguous()
    ws = torch.zeros(gq.workspace_size(B * T, C, S), dtype=torch.uint8, device=DEV)
    if paged:
        pt = inputs.paginate(t, page, extra_pages=2)
        out = gq.gqa_decode_paged(q4 if T > 1 else t["q"], pt["kv_pages"], pt["block_table"], pt["lens"],
                                  num_splits=S, workspace=ws, kv_scales=pt.get("kv_scale_pages"), **fp8)
    else:
        out = gq.gqa_decode_verify(q4, t["kv"], t["lens"], num_splits=S, workspace=ws, kv_scales=t["kv_scales"],
                                   **fp8)
    return t, out, ws


@pytest.mark.parametrize("kv_dtype", ["f16", "bf16", "e4m3", "i8"])
@pytest.mark.parametrize("T", [1, 2, 4])
@pytest.mark.parametrize("grid", ["balanced", "one piece", "cluster", "paged"])
def test_every_path(kv_dtype, T, grid):
    rng = np.random.default_rng(zlib.crc32(f"{kv_dtype}/{T}/{grid}".encode()))
    if grid == "balanced":    # more than one wave of pieces: the balanced schedule and the combine
        B, C, S = 96, 1024, 4
    elif grid == "one piece":  # many splits, one wave: one piece per CTA and the combine
        B, C, S = 2, 2048, 16
    elif grid == "cluster":   # 2-8 splits in one wave: merged on chip
        B, C, S = 2, 1024, 4
    else:
        B, C, S = 40, 1024, 4
    lens = rng.integers(T, C + 1, B)
    lens[0] = T
    lens[-1] = C
    if kv_dtype == "i8":
        lens[1 % B] = 8 * (C // 16) + 5  # a tail of row scales that are not a whole 16-byte group
    t, out, ws = _window(kv_dtype, B, C, T, lens.tolist(), S, paged=grid == "paged")
    _check(gq.get_status(ws), f"{kv_dtype} T={T} {grid}")
    ok, err, _ = tolerance_ok(_rows(out), _oracle(t))
    assert ok, f"{kv_dtype} T={T} {grid}: max err {err:.3e}"


@pytest.mark.parametrize("kv_dtype", ["f16", "e4m3", "i8"])
@pytest.mark.parametrize("T", [1, 3])
def test_capacity_off_the_tile_grid(kv_dtype, T):
    # one-piece grids (clusters, and with 9 splits the combine kernel) whose
    # last chunk, and the L2 prefetch of its first tile, end inside a tile
    for C, S in ((1000, 6), (1032, 5), (1032, 16)):
        lens = [C, C - 1, C // 2 + 3, T]
        t, out, ws = _window(kv_dtype, 4, C, T, lens, S)
        _check(gq.get_status(ws), f"{kv_dtype} T={T} C={C} S={S}")
        ok, err, _ = tolerance_ok(_rows(out), _oracle(t))
        assert ok, f"{kv_dtype} T={T} C={C} S={S}: max err {err:.3e}"


def test_out_of_contract_lengths_and_pages_are_clamped_not_out_of_range():
    B, C, T = 4, 512, 2
    t, _, ws = _window("bf16", B, C, T, [0, C + 9, 1, 300], 4)
    flags = gq.get_status(ws)
    assert flags & api.FLAG_LENGTH_CLAMPED
    _check(flags, "clamped lengths")
    w = inputs.custom(B, C, 300, kv_dtype="e4m3", kv_std=2.0)
    t = inputs.make(w, DEV)
    pt = inputs.paginate(t, 64, extra_pages=1)
    pt["block_table"][0, 1] = pt["num_pages"] + 7
    pt["block_table"][2, 0] = -3
    ws = torch.zeros(gq.workspace_size(B, C, 4), dtype=torch.uint8, device=DEV)
    gq.gqa_decode_paged(pt["q"], pt["kv_pages"], pt["block_table"], pt["lens"], k_scale=t["k_scale"],
                        v_scale=t["v_scale"], num_splits=4, workspace=ws)
    flags = gq.get_status(ws)
    assert flags & api.FLAG_PAGE_CLAMPED
    _check(flags, "clamped page ids")


def test_staged_calls():
    t = inputs.make(inputs.custom(3, 900, 50, 900, kv_dtype="e4m3", q_dtype="f16", kv_std=2.0, nan_tail=True), DEV)
    p = gq.prepare({"Q": t["q"], "KV": t["kv"], "O": torch.empty_like(t["q"]), "sequence_lengths": t["lens"]},
                   num_splits=5, k_scale=t["k_scale"], v_scale=t["v_scale"])
    gq.split_stage(p)
    gq.combine_stage(p)
    _check(gq.get_status(p), "staged calls")
    ok, err, _ = tolerance_ok(_rows(p.out), _oracle(t))
    assert ok, f"staged: max err {err:.3e}"


@pytest.mark.parametrize("fmt", ["bf16", "e4m3", "i8"])
@pytest.mark.parametrize("paged", [False, True])
def test_append(fmt, paged):
    B, C, page = 4, 512, 64
    g = torch.Generator(device=DEV)
    g.manual_seed(3)
    r = lambda *s: torch.randn(s, generator=g, device=DEV).to(torch.bfloat16)  # noqa: E731
    w = inputs.custom(B, C, 1, kv_dtype=fmt, q_dtype="bf16", kv_std=2.0 if fmt == "e4m3" else 1.0)
    t = inputs.make(w, DEV, lens=[100, 200, 300, 400])
    ks = t["k_scale"] if fmt == "e4m3" else 1.0
    vs = t["v_scale"] if fmt == "e4m3" else 1.0
    slots = torch.tensor([100, C + 4, 300, 400], dtype=torch.int32, device=DEV)  # one slot out of range
    pos = torch.arange(B, dtype=torch.int32, device=DEV) * 1000
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    if paged:
        pt = inputs.paginate(t, page, extra_pages=2)
        gq.append_kv_paged(r(B, 32, 128), r(B, 8, 128), r(B, 8, 128), r(128), r(128), pos, slots, pt["kv_pages"],
                           pt["block_table"], k_scale=ks, v_scale=vs, kv_scales=pt.get("kv_scale_pages"),
                           workspace=ws)
    else:
        gq.append_kv(r(B, 32, 128), r(B, 8, 128), r(B, 8, 128), r(128), r(128), pos, slots, t["kv"], k_scale=ks,
                     v_scale=vs, kv_scales=t["kv_scales"], workspace=ws)
    flags = gq.get_status(ws)
    assert flags & api.FLAG_SLOT_CLAMPED
    _check(flags, f"append {fmt} paged={paged}")


def test_no_allocation_entry():
    lib = _lib.load()
    t = inputs.make(inputs.WORKLOADS[3], DEV)
    out = torch.empty_like(t["q"])
    st = lib.gqa_decode_noalloc(t["q"].data_ptr(), t["kv"].data_ptr(), t["lens"].data_ptr(), out.data_ptr(), 32,
                                8192, 0, 1.0, 0, torch.cuda.current_stream(DEV).cuda_stream)
    assert st == 0, lib.gqa_last_error().decode()
    flags = ctypes.c_uint32(0)
    assert lib.gqa_decode_noalloc_get_status(torch.cuda.current_stream(DEV).cuda_stream, ctypes.byref(flags)) == 0
    _check(flags.value, "no-allocation entry")
    ok, err, _ = tolerance_ok(_rows(out), _oracle(t))
    assert ok, f"noalloc: max err {err:.3e}"


@pytest.mark.parametrize("case", ["bf16", "bf16 paged", "i8 scales"])
def test_cut_extents_make_the_checks_fire(case):
    """With the extents the checks compare against cut short, accesses past
    the cut must be reported (and redirected inside the real buffers, so
    nothing faults); with the true extents restored the same call is clean
    and matches the oracle."""
    lib = _lib.load()
    kv_dtype = "i8" if case.startswith("i8") else "bf16"
    B, C, S = 4, 1024, 4
    lens = [C, 700, C, 8 * (C // 16) + 5]  # the last: a tail of int8 scales loaded one by one
    w = inputs.custom(B, C, 1, kv_dtype=kv_dtype)
    t = inputs.make(w, DEV, lens=lens)
    kv_bytes = t["kv"].numel() * t["kv"].element_size()
    sc_bytes = t["kv_scales"].numel() * 2 if t["kv_scales"] is not None else 0

    def run():
        ws = torch.zeros(gq.workspace_size(B, C, S), dtype=torch.uint8, device=DEV)
        if case.endswith("paged"):
            pt = inputs.paginate(t, 64, extra_pages=2)
            out = gq.gqa_decode_paged(t["q"], pt["kv_pages"], pt["block_table"], pt["lens"], num_splits=S,
                                      workspace=ws)
        else:
            out = gq.gqa_decode_verify(t["q"][:, None].contiguous(), t["kv"], t["lens"], num_splits=S, workspace=ws,
                                       kv_scales=t["kv_scales"])
        torch.cuda.synchronize(DEV)
        return out, gq.get_status(ws)

    try:
        if case.startswith("i8"):
            assert lib.gqa_decode_debug_cut_extents(0, sc_bytes // 2) == 0
        else:
            assert lib.gqa_decode_debug_cut_extents(kv_bytes // 2, 0) == 0
        _, flags = run()
        assert flags & FLAG_BOUNDS, f"{case}: the cut extent was not reported (flags {flags:#x})"
        assert not flags & api.FLAG_WAIT_TIMEOUT
    finally:
        assert lib.gqa_decode_debug_cut_extents(0, 0) == 0
    out, flags = run()
    _check(flags, f"{case}, true extents")
    ok, err, _ = tolerance_ok(_rows(out), _oracle(t))
    assert ok, f"{case}: max err {err:.3e}"
