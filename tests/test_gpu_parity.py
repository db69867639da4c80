"""GPU parity: the CUDA path (through the C ABI) against the FP64 oracle.

Bar (element-wise): |gpu - oracle| <= 3e-3, or <= 1e-2 * |oracle| where
|oracle| > 0.3, every output finite.  Small workloads are compared on every
element; the two full-size workloads (bf16 8 x 131072, e4m3 64 x U[16k,32k])
are run in the launch configuration the benchmark times and compared on
sampled (b, KV head) units (all 4 query heads each).  Also covered: ragged
lengths and tile edges, capacity 1, every split count, q_scale 0, distinct
fp8 scales, NaN tails (bit-exact output whatever the unused slots hold; the
cache is never written), guard bands around the output and the workspace,
run-to-run determinism, CUDA-graph capture and replay (the prepared call, the
append + decode serving step, the paged, int8 and verify entry points), length
clamping flags, the convenience and staged entry points, errors reported
before launch, and the balanced schedule's edge cases.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
import gqa_decode_attention_sm_gb300 as gq
from gqa_decode_attention_sm_gb300 import _lib, api, inputs
from helpers import HQ, RMS_GATE, bits_of, rms_gate_ok, tolerance_ok, ulps_apart

pytestmark = pytest.mark.gpu

FMT = {"f16": oracle.F16, "bf16": oracle.BF16, "e4m3": oracle.E4M3, "i8": oracle.I8}
DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gqa_decode_attention_sm_gb300 import build as gbuild
    gbuild.build()
    oracle.build()
    torch.cuda.init()


def _make(w, **kw):
    return inputs.make(w, DEV, **kw)


def _prepare(t, out=None, num_splits=None, workspace=None):
    w = t["workload"]
    out = torch.empty_like(t["q"]) if out is None else out
    fp8 = w.kv_dtype == "e4m3"
    tensors = {"Q": t["q"], "KV": t["kv"], "O": out, "sequence_lengths": t["lens"]}
    if t.get("kv_scales") is not None:
        tensors["KV_SCALES"] = t["kv_scales"]
    return gq.prepare(tensors,
                      q_scale=t["q_scale"], num_splits=num_splits,
                      k_scale=t["k_scale"] if fp8 else None, v_scale=t["v_scale"] if fp8 else None,
                      workspace=workspace)


def _run(t, num_splits=None):
    p = _prepare(t, num_splits=num_splits)
    gq.launch(p)
    torch.cuda.synchronize()
    return p


def _oracle_full(t, **kw):
    w = t["workload"]
    args = dict(q_scale=t["q_scale"], k_scale=t["k_scale"], v_scale=t["v_scale"])
    if t.get("kv_scales") is not None:
        args["kv_scales"] = bits_of(t["kv_scales"])
    args.update(kw)
    out, _ = oracle.gqa_decode(bits_of(t["q"]), FMT[w.q_dtype], bits_of(t["kv"]), FMT[w.kv_dtype],
                               t["lens"].cpu().numpy(), **args)
    return out


def _oracle_units(t, units):
    """Oracle rows for sampled (b, g) units: copies only those K/V planes to the host."""
    w = t["workload"]
    C = w.capacity
    lens = t["lens"].cpu().numpy()
    res = {}
    for b, g in units:
        qb = bits_of(t["q"][b:b + 1])
        kvb = np.zeros((1, 2, 8, C, 128), dtype=np.uint8 if w.kv_dtype in ("e4m3", "i8") else np.uint16)
        kvb[0, :, g] = bits_of(t["kv"][b, :, g])
        extra = {}
        if t.get("kv_scales") is not None:
            scb = np.zeros((1, 2, 8, C), dtype=np.uint16)
            scb[0, :, g] = bits_of(t["kv_scales"][b, :, g])
            extra["kv_scales"] = scb
        rows = [4 * g + j for j in range(4)]
        out, _ = oracle.gqa_decode(qb, FMT[w.q_dtype], kvb, FMT[w.kv_dtype], lens[b:b + 1],
                                   q_scale=t["q_scale"], k_scale=t["k_scale"],
                                   v_scale=t["v_scale"], rows=rows, **extra)
        for j, r in enumerate(rows):
            res[b * HQ + r] = out[j]
    return res


def _gpu_rows(out):
    return out.float().cpu().numpy().reshape(-1, 128)


def _assert_parity(got, ref, what="", rms_gate=False):
    """The element-wise bar; with ``rms_gate`` also max |err| <= 0.05 RMS(ref)
    (long contexts, where the absolute bar is most of the signal)."""
    ok, err, excess = tolerance_ok(got, ref)
    gate_ok, ratio = rms_gate_ok(got, ref)
    print(f"PARITY {what}: max|err| {err:.3e}, max err / rms(ref) {ratio:.3e}")
    assert ok, f"{what}: max |gpu - oracle| {err:.3e} exceeds the bar by {excess:.3e}"
    if rms_gate:
        assert gate_ok, f"{what}: max |gpu - oracle| is {ratio:.3e} of RMS(oracle), above {RMS_GATE}"


# ---------------------------------------------------------------- workloads


@pytest.mark.parametrize("index", [1, 2, 3])
def test_workload_every_element(index):
    t = _make(inputs.WORKLOADS[index])
    p = _run(t)
    _assert_parity(_gpu_rows(p.out), _oracle_full(t), f"workload {index} (splits {p.num_splits})",
                   rms_gate=True)


@pytest.mark.parametrize("index", [4, 5])
def test_full_size_workload_sampled(index):
    w = inputs.WORKLOADS[index]
    t = _make(w)
    p = _run(t)  # the auto plan: the launch configuration the benchmark times
    rng = np.random.default_rng(index)
    units = sorted({(int(b), int(g)) for b, g in zip(rng.integers(0, w.batch, 6), rng.integers(0, 8, 6))}
                   | {(0, 0), (w.batch - 1, 7)})
    ref = _oracle_units(t, units)
    got = _gpu_rows(p.out)
    rows = sorted(ref)
    _assert_parity(got[rows], np.stack([ref[r] for r in rows]), f"workload {index} sampled", rms_gate=True)
    assert np.isfinite(got).all()


def _oracle_units_window(t, units):
    """Oracle rows of sampled (b, g) units for every query token of a window."""
    w = t["workload"]
    T, C = w.q_len, w.capacity
    lens = t["lens"].cpu().numpy()
    res = {}
    for b, g in units:
        kvb = np.zeros((1, 2, 8, C, 128), dtype=np.uint8 if w.kv_dtype in ("e4m3", "i8") else np.uint16)
        kvb[0, :, g] = bits_of(t["kv"][b, :, g])
        rows = [jt * HQ + 4 * g + j for jt in range(T) for j in range(4)]
        out, _ = oracle.gqa_decode(bits_of(t["q"][b:b + 1]), FMT[w.q_dtype], kvb, FMT[w.kv_dtype], lens[b:b + 1],
                                   q_scale=t["q_scale"], k_scale=t["k_scale"], v_scale=t["v_scale"], rows=rows)
        for k, r in enumerate(rows):
            res[b * T * HQ + r] = out[k]
    return res


def test_full_size_verify_window_sampled():
    # workload 4 with a 2-token window, in the launch configuration the benchmark times
    w = inputs.with_(inputs.WORKLOADS[4], q_len=2)
    t = _make(w)
    out = _verify(t)
    ref = _oracle_units_window(t, [(0, 0), (3, 5), (7, 7)])
    rows = sorted(ref)
    _assert_parity(_gpu_rows(out)[rows], np.stack([ref[r] for r in rows]), "workload 4, window 2, sampled",
                   rms_gate=True)


def test_full_size_fp8_verify_window_sampled():
    # workload 5 (e4m3 KV) with a 2-token window, as the per-workload table times
    # it: 8-bit 2-token windows run 3 CTAs of 2 stages per SM
    w = inputs.with_(inputs.WORKLOADS[5], q_len=2)
    t = _make(w)
    S = gq.plan(w.batch, w.capacity, 2, DEV)
    out = _verify(t, num_splits=S)
    ref = _oracle_units_window(t, [(0, 0), (29, 4), (63, 7)])
    rows = sorted(ref)
    _assert_parity(_gpu_rows(out)[rows], np.stack([ref[r] for r in rows]), "workload 5, window 2, sampled",
                   rms_gate=True)


@pytest.mark.parametrize("kv_dtype,T", [("e4m3", 3), ("i8", 4)])
def test_full_size_8bit_long_window_sampled(kv_dtype, T):
    # 3- and 4-token windows over an 8-bit cache of workload 5's shape, as the
    # per-workload table times them: the balanced schedule, two mma n-tiles,
    # 2 CTAs of 3 stages per SM
    base = inputs.WORKLOADS[5] if kv_dtype == "e4m3" else inputs.custom(64, 32768, 16384, 32768, kv_dtype="i8",
                                                                          index=5)
    w = inputs.with_(base, q_len=T)
    t = _make(w)
    fmt = {"e4m3": 2, "i8": 3}[kv_dtype]
    out = _verify(t, num_splits=gq.plan(w.batch, w.capacity, fmt, DEV))
    units = [(0, 0), (21, 6), (63, 7)]
    ref = {}
    for b, g in units:
        kvb = np.zeros((1, 2, 8, w.capacity, 128), dtype=np.uint8)
        kvb[0, :, g] = bits_of(t["kv"][b, :, g])
        extra = {}
        if t.get("kv_scales") is not None:
            scb = np.zeros((1, 2, 8, w.capacity), dtype=np.uint16)
            scb[0, :, g] = bits_of(t["kv_scales"][b, :, g])
            extra["kv_scales"] = scb
        rows = [jt * HQ + 4 * g + j for jt in range(T) for j in range(4)]
        o, _ = oracle.gqa_decode(bits_of(t["q"][b:b + 1]), FMT[w.q_dtype], kvb, FMT[kv_dtype],
                                 t["lens"].cpu().numpy()[b:b + 1], q_scale=t["q_scale"], k_scale=t["k_scale"],
                                 v_scale=t["v_scale"], rows=rows, **extra)
        for k, r in enumerate(rows):
            ref[b * T * HQ + r] = o[k]
    rows = sorted(ref)
    _assert_parity(_gpu_rows(out)[rows], np.stack([ref[r] for r in rows]),
                   f"{kv_dtype} 64 x U[16k,32k], window {T}, sampled", rms_gate=True)
    assert np.isfinite(_gpu_rows(out)).all()


def test_full_size_paged_int8_sampled():
    # the int8 cache of workload 5's shape in shuffled 256-token pages, as benchmarked
    w = inputs.custom(64, 32768, 16384, 32768, kv_dtype="i8", index=5)
    t = _make(w)
    units = [(0, 0), (17, 3), (63, 7)]
    ref = _oracle_units(t, units)
    pt = inputs.paginate(t, 256, extra_pages=8)
    del t["kv"]
    out = _paged(pt)
    torch.cuda.synchronize()
    rows = sorted(ref)
    _assert_parity(_gpu_rows(out)[rows], np.stack([ref[r] for r in rows]), "paged int8 full size, sampled",
                   rms_gate=True)


# ---------------------------------------------------------------- edge cases


@pytest.mark.parametrize("kv_dtype", ["f16", "bf16", "e4m3", "i8"])
def test_tile_edges_and_ragged_lengths(kv_dtype):
    lens = [1, 2, 63, 64, 65, 127, 128, 129, 255, 256, 200, 17]
    w = inputs.custom(len(lens), 256, 1, kv_dtype=kv_dtype, kv_std=2.0 if kv_dtype == "e4m3" else 1.0,
                      nan_tail=True)
    t = _make(w, lens=lens)
    for S in (None, 1, 3):
        p = _run(t, num_splits=S)
        _assert_parity(_gpu_rows(p.out), _oracle_full(t), f"{kv_dtype} edges splits={p.num_splits}")


def test_capacity_one():
    t = _make(inputs.custom(5, 1, 1))
    p = _run(t)
    got = _gpu_rows(p.out)
    _assert_parity(got, _oracle_full(t), "capacity 1")
    # one slot: the output is V[0] itself, exactly
    v0 = t["kv"][:, 1, :, 0, :].float().cpu().numpy()  # [B,8,128]
    assert np.array_equal(got.reshape(5, 32, 128), np.repeat(v0, 4, axis=1))


@pytest.mark.parametrize("kv_dtype", ["f16", "e4m3", "i8"])
@pytest.mark.parametrize("S", [1, 2, 3, 7, 16, 64, 256])
def test_every_split_count(kv_dtype, S):
    w = inputs.custom(3, 1000, 1, kv_dtype=kv_dtype, kv_std=2.0 if kv_dtype == "e4m3" else 1.0,
                      nan_tail=True)
    t = _make(w, lens=[1000, 333, 1])
    p = _run(t, num_splits=S)
    _assert_parity(_gpu_rows(p.out), _oracle_full(t), f"{kv_dtype} splits={S}")


@pytest.mark.parametrize("q_dtype", ["bf16", "f16"])
def test_int8_every_element(q_dtype):
    t = _make(inputs.custom(6, 1024, 1, 1024, kv_dtype="i8", q_dtype=q_dtype, nan_tail=True))
    for S in (None, 1, 5):
        p = _run(t, num_splits=S)
        _assert_parity(_gpu_rows(p.out), _oracle_full(t), f"int8 KV, {q_dtype} q, splits={p.num_splits}")


@pytest.mark.parametrize("q_dtype,shift,q_scale", [("bf16", 8.0, 2.0), ("f16", 3.0, 4.0)])
def test_int8_large_q_sum_sharp_softmax(q_dtype, shift, q_scale):
    # int8 K enters the tensor core as code + 1152 and the scores take
    # 1152 * sum_d q_d back off: q with a large mean (a large sum) and a sharp
    # softmax make that difference as large as it gets relative to the scores
    w = inputs.custom(4, 4096, 1, 4096, kv_dtype="i8", q_dtype=q_dtype, index=90, q_scale=q_scale)
    t = _make(w)
    t["q"] = (t["q"].float() + shift).to(t["q"].dtype)
    for S in (None, 1):
        p = _run(t, num_splits=S)
        _assert_parity(_gpu_rows(p.out), _oracle_full(t), f"int8, q + {shift}, q_scale {q_scale}, splits={S}")


@pytest.mark.parametrize("kv_dtype", ["e4m3", "i8"])
@pytest.mark.parametrize("T", [1, 3])
@pytest.mark.parametrize("case", ["huge", "tiny", "mixed"])
def test_8bit_cache_takes_a_bf16_q_of_any_magnitude(kv_dtype, T, case):
    # 8-bit caches run on f16 tensor cores, whose range (6e-8 .. 65504) a bf16
    # q can leave; each query column is scaled by a power of two before its
    # conversion, so q is taken exactly.  huge: |q| ~ 1e6 (a near one-hot
    # softmax; saturating at 65504 would change which token wins).  tiny:
    # |q| ~ 1e-7 with q_scale 2e7 (an ordinary softmax of q values below the
    # f16 normal range).  mixed: head h at 10^(-7 + 13h/31), and element 0 of
    # every vector 1e3 times its neighbours.  T = 3 runs two mma n-tiles.
    B, C = 4, 704  # an int8 cache takes capacities that are multiples of 8
    w = inputs.custom(B, C, 1, kv_dtype=kv_dtype, kv_std=2.0 if kv_dtype == "e4m3" else 1.0, nan_tail=True,
                      q_len=T)
    t = _make(w, lens=[T, 129, 500, 700])
    g = torch.Generator(device=DEV)
    g.manual_seed(7)
    q = torch.randn(t["q"].shape, generator=g, device=DEV, dtype=torch.float32)
    q_scale = 1.0
    if case == "huge":
        q *= 1e6
    elif case == "tiny":
        q *= 1e-7
        q_scale = 2e7
    else:
        q *= (10.0 ** torch.linspace(-7, 6, HQ, device=DEV)).view(HQ, 1)
        q[..., 0] *= 1e3
    t["q"] = q.to(torch.bfloat16)
    t["q_scale"] = q_scale
    for S in (None, 1):
        out = _verify(t, num_splits=S)
        _assert_parity(_gpu_rows(out), _oracle_full(t), f"{kv_dtype} T={T} bf16 q {case} splits={S}")


def test_int8_full_size_sampled():
    # the e4m3 workload's shape and length mix with an int8 cache (4.3 GB of codes)
    w = inputs.custom(64, 32768, 16384, 32768, kv_dtype="i8", index=5)
    t = _make(w)
    p = _run(t)
    units = [(0, 0), (17, 3), (40, 6), (63, 7)]
    ref = _oracle_units(t, units)
    rows = sorted(ref)
    _assert_parity(_gpu_rows(p.out)[rows], np.stack([ref[r] for r in rows]), "int8 64 x U[16k,32k] sampled",
                   rms_gate=True)


def test_bf16_every_element_multi_split():
    t = _make(inputs.custom(2, 4096, 4096, kv_dtype="bf16"))
    p = _run(t)
    assert p.num_splits > 1
    _assert_parity(_gpu_rows(p.out), _oracle_full(t), "bf16 2x4096")


def test_q_scale_zero_gives_mean_through_convenience_call():
    w = inputs.custom(2, 500, 100, 500)
    t = _make(w)
    out = gq.gqa_decode(t["q"], t["kv"], t["lens"], q_scale=0.0)
    torch.cuda.synchronize()
    _assert_parity(_gpu_rows(out), _oracle_full(t, q_scale=0.0), "q_scale=0")


def test_large_q_scale_peaky_softmax():
    w = inputs.custom(2, 700, 300, 700, q_scale=8.0)
    t = _make(w)
    p = _run(t)
    _assert_parity(_gpu_rows(p.out), _oracle_full(t), "q_scale=8")


def test_fp8_distinct_scales():
    w = inputs.custom(4, 2048, 500, 2048, kv_dtype="e4m3", kv_std=2.0)
    t = _make(w)
    t["k_scale"] *= 0.5
    t["v_scale"] *= 3.0
    p = _run(t)
    _assert_parity(_gpu_rows(p.out), _oracle_full(t), "fp8 k_scale != v_scale")


def test_fp8_with_f16_query_through_stages():
    w = inputs.custom(3, 900, 50, 900, kv_dtype="e4m3", q_dtype="f16", kv_std=2.0, nan_tail=True)
    t = _make(w)
    p = _prepare(t, num_splits=4)
    gq.split_stage(p)
    gq.combine_stage(p)
    torch.cuda.synchronize()
    _assert_parity(_gpu_rows(p.out), _oracle_full(t), "e4m3 KV, f16 q")


def test_large_batch_small_capacity():
    t = _make(inputs.custom(4096, 64, 1, 64))
    p = _run(t)
    _assert_parity(_gpu_rows(p.out), _oracle_full(t), "B=4096 C=64")


def test_max_batch():
    # 65535 rows, the largest batch the ABI takes (the one-piece grid's y limit)
    B = 65535
    rng = np.random.default_rng(65535)
    t = _make(inputs.custom(B, 16, 1, 16), lens=rng.integers(1, 17, B).tolist())
    p = _run(t)
    _assert_parity(_gpu_rows(p.out), _oracle_full(t), "B=65535 C=16")


def test_max_capacity_sampled():
    w = inputs.custom(1, 1 << 20, 1 << 20, kv_dtype="bf16")
    t = _make(w)
    for S in (None, 256):
        p = _run(t, num_splits=S)
        ref = _oracle_units(t, [(0, 0), (0, 5)])
        rows = sorted(ref)
        _assert_parity(_gpu_rows(p.out)[rows], np.stack([ref[r] for r in rows]),
                       f"C=2^20 splits={p.num_splits}", rms_gate=True)


def test_long_request_sampled():
    # one long request (bf16, batch 1, 131072 tokens), in the launch
    # configuration the benchmark times: every KV head's row is cut into ~38
    # pieces by the balanced schedule and merged by the combine kernel
    w = inputs.custom(1, 131072, 131072, kv_dtype="bf16", index=4)
    t = _make(w)
    p = _run(t)
    ref = _oracle_units(t, [(0, 0), (0, 2), (0, 5), (0, 7)])
    rows = sorted(ref)
    _assert_parity(_gpu_rows(p.out)[rows], np.stack([ref[r] for r in rows]),
                   f"bf16 1 x 131072 splits={p.num_splits}", rms_gate=True)


# ------------------------------------------- balanced schedule (many waves)
#
# Grids of more than one wave of (split, KV head, batch row) work items run
# the balanced schedule: one CTA per resident slot, each taking an equal run
# of the tiles of all rows (lengths read on the device), rows cut into pieces
# wherever the runs end.  These cases are all well past one wave.


@pytest.mark.parametrize("kv_dtype", ["f16", "bf16", "e4m3", "i8"])
@pytest.mark.parametrize("S", [None, 2, 16])
def test_balanced_ragged_every_element(kv_dtype, S):
    rng = np.random.default_rng(7)
    C = 2048
    lens = rng.integers(1, C + 1, 96)
    lens[:6] = [1, 64, 128, 129, C, C - 1]  # tile edges of both tile sizes, full rows
    w = inputs.custom(96, C, 1, kv_dtype=kv_dtype, kv_std=2.0 if kv_dtype == "e4m3" else 1.0, nan_tail=True)
    t = _make(w, lens=lens.tolist())
    p = _run(t, num_splits=S)
    _assert_parity(_gpu_rows(p.out), _oracle_full(t), f"balanced {kv_dtype} splits={p.num_splits}")


def test_balanced_zero_length_rows_and_all_zero():
    C, B = 2048, 64
    lens = [0 if b % 3 == 0 else (b * 97) % C + 1 for b in range(B)]
    t = _make(inputs.custom(B, C, 1), lens=lens)
    p = _run(t, num_splits=8)
    assert gq.get_status(p) & api.FLAG_LENGTH_CLAMPED
    out = p.out.view(B, 32, 128)
    zero = [b for b in range(B) if lens[b] == 0]
    keep = [b for b in range(B) if lens[b] > 0]
    assert not out[zero].any()
    sub = dict(t, q=t["q"][keep], kv=t["kv"][keep], lens=t["lens"][keep])
    _assert_parity(_gpu_rows(out[keep]), _oracle_full(sub), "balanced, zero-length rows")
    t["lens"].zero_()
    p.out.fill_(1.0)
    gq.launch(p)
    torch.cuda.synchronize()
    assert not p.out.any()


def test_balanced_one_long_row_among_short_ones():
    # one row holds almost all the tiles: runs are cut by the split-slot bound
    C, B = 65536, 64
    lens = [C] + [1 + 5 * b for b in range(1, B)]
    t = _make(inputs.custom(B, C, 1, kv_dtype="bf16"), lens=lens)
    for S in (None, 4):
        p = _run(t, num_splits=S)
        _assert_parity(_gpu_rows(p.out), _oracle_full(t), f"one long row, splits={p.num_splits}")


@pytest.mark.parametrize("B,L,kv_dtype", [(16, 8192, "bf16"), (256, 1000, "f16"), (96, 3000, "e4m3")])
def test_balanced_uniform_rows(B, L, kv_dtype):
    # equal lengths: rows at least one CTA's run long are cut without the
    # per-row piece cost (16 x 8192), shorter ones with it (256 x 1000,
    # 96 x 3000); both kernels take the same choice from the lengths
    w = inputs.custom(B, L, L, kv_dtype=kv_dtype, kv_std=2.0 if kv_dtype == "e4m3" else 1.0)
    t = _make(w)
    p = _run(t, num_splits=8)
    _assert_parity(_gpu_rows(p.out), _oracle_full(t), f"uniform {B} x {L} {kv_dtype}")


@pytest.mark.parametrize("B", [1024, 1025])
def test_balanced_batch_limit(B):
    # 1024 rows is the largest batch the balanced prologue scans; 1025 runs the
    # one-piece-per-CTA grid
    rng = np.random.default_rng(B)
    t = _make(inputs.custom(B, 256, 1), lens=rng.integers(1, 257, B).tolist())
    p = _run(t, num_splits=4)
    _assert_parity(_gpu_rows(p.out), _oracle_full(t), f"B={B}")


@pytest.mark.parametrize("kv_dtype", ["f16", "e4m3"])
def test_balanced_paged_ragged(kv_dtype):
    rng = np.random.default_rng(11)
    C = 4096
    w = inputs.custom(48, C, 1, kv_dtype=kv_dtype, kv_std=2.0 if kv_dtype == "e4m3" else 1.0, nan_tail=True)
    t = _make(w, lens=rng.integers(1, C + 1, 48).tolist())
    ref = _oracle_full(t)
    pt = inputs.paginate(t, 256, extra_pages=5)
    out = _paged(pt, num_splits=8)
    torch.cuda.synchronize()
    _assert_parity(_gpu_rows(out), ref, f"balanced paged {kv_dtype}")


# ------------------------------------------------------ unused slots, safety


@pytest.mark.parametrize("kv_dtype", ["f16", "e4m3", "i8"])
def test_output_bit_exact_whatever_the_unused_slots_hold(kv_dtype):
    w = inputs.custom(6, 640, 1, 600, kv_dtype=kv_dtype, kv_std=2.0 if kv_dtype == "e4m3" else 1.0)
    t = _make(w)
    outs = []
    for fill in (float("nan"), 0.0, 300.0):
        kv = t["kv"].clone()
        inputs.fill_tail(kv, t["lens"], kv_dtype, fill)
        before = kv.clone()
        t2 = dict(t, kv=kv)
        if kv_dtype == "i8":  # the unused rows' scales too
            sc = t["kv_scales"].clone()
            for b, L in enumerate(t["lens"].tolist()):
                sc[b, :, :, L:] = fill
            t2["kv_scales"] = sc
        for S in (1, 5):
            p = _run(t2, num_splits=S)
            outs.append((S, p.out.clone()))
        assert torch.equal(kv.view(torch.uint8), before.view(torch.uint8)), "the cache was written"
    for S in (1, 5):
        same = [o for s, o in outs if s == S]
        for o in same[1:]:
            assert torch.equal(o.view(torch.int16), same[0].view(torch.int16))


def test_guard_bands_untouched():
    w = inputs.custom(3, 512, 100, 512)
    t = _make(w)
    G = 4096
    out_buf = torch.full((G + 3 * 32 * 128 + G,), 0x5A5A, dtype=torch.int16, device=DEV)
    out = out_buf[G:G + 3 * 32 * 128].view(torch.float16).view(3, 32, 128)
    S = 6
    nws = gq.workspace_size(3, 512, S)
    ws_buf = torch.full((G + nws + G,), 0xA5, dtype=torch.uint8, device=DEV)
    ws = ws_buf[G:G + nws]
    ws[:256].zero_()
    p = _prepare(t, out=out, num_splits=S, workspace=ws)
    gq.launch(p)
    torch.cuda.synchronize()
    assert bool((out_buf[:G] == 0x5A5A).all() and (out_buf[-G:] == 0x5A5A).all())
    assert bool((ws_buf[:G] == 0xA5).all() and (ws_buf[-G:] == 0xA5).all())
    _assert_parity(_gpu_rows(out), _oracle_full(t), "guarded")


def test_deterministic_across_runs():
    t = _make(inputs.WORKLOADS[3])
    p = _prepare(t)
    first = gq.launch(p).clone()
    for _ in range(3):
        assert torch.equal(gq.launch(p).view(torch.int16), first.view(torch.int16))


@pytest.mark.parametrize("kv_dtype", ["f16", "bf16", "e4m3", "i8"])
@pytest.mark.parametrize("T", [1, 2, 4])
@pytest.mark.parametrize("grid", ["balanced", "cluster", "combine", "paged"])
def test_determinism_soak(kv_dtype, T, grid):
    # 16 launches back to back, no synchronisation between them, each output
    # copied off on the stream: every one bitwise equal to the first.  A race
    # in a merge area shared between a CTA's pieces, between the ring and the
    # epilogue, or between cluster members would show as a differing bit.
    B, C, S = {"balanced": (96, 2048, 4), "cluster": (2, 1024, 4), "combine": (2, 2048, 16),
               "paged": (64, 2048, 4)}[grid]
    rng = np.random.default_rng(zlib.crc32(f"{kv_dtype}/{T}/{grid}".encode()))
    lens = rng.integers(T, C + 1, B).tolist()
    w = inputs.custom(B, C, 1, kv_dtype=kv_dtype, kv_std=2.0 if kv_dtype == "e4m3" else 1.0, nan_tail=True,
                      q_len=T)
    t = _make(w, lens=lens)
    fp8 = dict(k_scale=t["k_scale"], v_scale=t["v_scale"]) if kv_dtype == "e4m3" else {}
    q4 = t["q"] if T > 1 else t["q"][:, None].contiguous()
    ws = torch.zeros(gq.workspace_size(B * T, C, S), dtype=torch.uint8, device=DEV)
    if grid == "paged":
        pt = inputs.paginate(t, 64, extra_pages=2)
        run = lambda: gq.gqa_decode_paged(q4 if T > 1 else t["q"], pt["kv_pages"], pt["block_table"],  # noqa: E731
                                          pt["lens"], num_splits=S, workspace=ws,
                                          kv_scales=pt.get("kv_scale_pages"), **fp8)
    else:
        run = lambda: gq.gqa_decode_verify(q4, t["kv"], t["lens"], num_splits=S, workspace=ws,  # noqa: E731
                                           kv_scales=t["kv_scales"], **fp8)
    outs = [run().clone() for _ in range(16)]
    torch.cuda.synchronize()
    first = outs[0].view(torch.int16)
    for i, o in enumerate(outs[1:], 1):
        assert torch.equal(o.view(torch.int16), first), f"{kv_dtype} T={T} {grid}: launch {i} differs"
    assert not gq.get_status(ws) & (api.FLAG_WAIT_TIMEOUT | api.FLAG_LENGTH_CLAMPED)


def test_host_threads_launch_concurrently():
    # Four host threads, each with its own stream and prepared problem
    # (different formats and schedules), launch 10 times each while a fifth
    # thread makes calls that fail validation.  The library's shared state
    # (device set-up, the per-device tables) is guarded and its last-error
    # string is per thread: every output equals its sequential run bit for
    # bit, and each failing call reads its own message.
    import threading
    problems = [
        _make(inputs.custom(48, 2048, 1, 2048)),                                   # fp16, balanced
        _make(inputs.custom(2, 1024, 1024, kv_dtype="bf16")),                        # bf16, cluster merge
        _make(inputs.custom(64, 4096, 1024, 4096, kv_dtype="e4m3", kv_std=2.0)),    # e4m3, balanced
        _make(inputs.custom(8, 4096, 1024, 4096, kv_dtype="i8")),                   # int8, balanced
    ]
    preps = [_prepare(t) for t in problems]
    refs = [gq.launch(p).clone() for p in preps]
    torch.cuda.synchronize()
    for p in preps:
        p.out.zero_()
    errors, failures = [], []
    start = threading.Barrier(5)

    def worker(i):
        try:
            s = torch.cuda.Stream()
            start.wait()
            with torch.cuda.stream(s):
                for _ in range(10):
                    gq.launch(preps[i])
            s.synchronize()
        except Exception as e:  # noqa: BLE001 - reported below
            errors.append(f"thread {i}: {e!r}")

    def failing():
        lib = _lib.load()
        start.wait()
        for k in range(200):
            st = lib.gqa_decode_prepared(None, None, None, None, 1, 64 + k, 0, 1.0, 1, None, 0, None)
            msg = lib.gqa_last_error().decode()
            if st == 0 or "null" not in msg:
                failures.append((st, msg))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(4)] + [threading.Thread(target=failing)]
    for th in threads:
        th.start()
    for th in threads:
        th.join(timeout=120)
    assert not errors, errors
    assert not failures, failures[:3]
    torch.cuda.synchronize()
    for i, (p, ref) in enumerate(zip(preps, refs)):
        assert torch.equal(p.out.view(torch.int16), ref.view(torch.int16)), f"problem {i} differs"


def test_concurrent_streams_with_their_own_workspaces():
    # Launches on different streams with distinct workspaces may overlap on
    # the GPU: nothing in the library is shared between them.  Two problems
    # on two streams, launched alternately with no synchronisation between
    # them, each give the output of their sequential run bit for bit.
    ta = _make(inputs.WORKLOADS[3])                                   # fp16, balanced grid + combine
    tb = _make(inputs.custom(6, 2048, 900, 2048, kv_dtype="e4m3", kv_std=2.0, q_len=3))  # e4m3 window
    pa = _prepare(ta)
    ref_a = gq.launch(pa).clone()
    fp8 = dict(k_scale=tb["k_scale"], v_scale=tb["v_scale"])
    wsb = torch.zeros(gq.workspace_size(6 * 3, 2048, 4), dtype=torch.uint8, device=DEV)
    out_b = torch.empty_like(tb["q"])

    def run_b():
        gq.gqa_decode_verify(tb["q"], tb["kv"], tb["lens"], out=out_b, num_splits=4, workspace=wsb, **fp8)

    run_b()
    torch.cuda.synchronize()
    ref_b = out_b.clone()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    sa.wait_stream(torch.cuda.current_stream())
    sb.wait_stream(torch.cuda.current_stream())
    for _ in range(8):
        with torch.cuda.stream(sa):
            gq.launch(pa)
        with torch.cuda.stream(sb):
            run_b()
    torch.cuda.synchronize()
    assert torch.equal(pa.out.view(torch.int16), ref_a.view(torch.int16))
    assert torch.equal(out_b.view(torch.int16), ref_b.view(torch.int16))
    _assert_parity(_gpu_rows(out_b), _oracle_full(tb), "e4m3 3-token window after concurrent launches")


def test_graph_capture_replay_matches_eager():
    w = inputs.custom(4, 4096, 1000, 4096)
    t = _make(w)
    p = _prepare(t)
    eager = gq.launch(p).clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        gq.launch(p)  # warm-up on a side stream before capture
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        gq.launch(p)
    p.out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(p.out.view(torch.int16), eager.view(torch.int16))
    # update the lengths in place (same address) and replay
    t["lens"].fill_(777)
    g.replay()
    torch.cuda.synchronize()
    replayed = p.out.clone()
    assert torch.equal(replayed.view(torch.int16), gq.launch(p).view(torch.int16))
    _assert_parity(_gpu_rows(replayed), _oracle_full(t), "graph replay, lengths 777")


def test_convenience_and_stages_match_prepared_bitwise():
    t = _make(inputs.WORKLOADS[2])
    p = _run(t)
    conv = gq.gqa_decode(t["q"], t["kv"], t["lens"])
    out2 = torch.empty_like(t["q"])
    p2 = _prepare(t, out=out2)
    gq.split_stage(p2)
    gq.combine_stage(p2)
    torch.cuda.synchronize()
    assert torch.equal(conv.view(torch.int16), p.out.view(torch.int16))
    assert torch.equal(out2.view(torch.int16), p.out.view(torch.int16))


@pytest.mark.parametrize("S", [1, 4])
def test_out_of_range_lengths_are_clamped_and_flagged(S):
    C = 256
    w = inputs.custom(3, C, 5)
    t = _make(w, lens=[0, C + 7, 5])
    p = _prepare(t, num_splits=S)
    assert gq.get_status(p) == 0
    gq.launch(p)
    flags = gq.get_status(p)
    assert flags & api.FLAG_LENGTH_CLAMPED and not flags & api.FLAG_WAIT_TIMEOUT
    assert gq.get_status(p) == 0  # read-and-clear
    got = p.out.clone()
    assert torch.all(got[0] == 0)
    t["lens"].copy_(torch.tensor([1, C, 5], dtype=torch.int32))
    gq.launch(p)
    torch.cuda.synchronize()
    assert torch.equal(got[1:].view(torch.int16), p.out[1:].view(torch.int16))
    assert gq.get_status(p) == 0


@pytest.mark.parametrize("kv_dtype", ["f16", "bf16", "e4m3", "i8"])
@pytest.mark.parametrize("C,S", [(1000, 6), (1032, 5), (1032, 16), (200, 3)])
def test_capacity_off_the_tile_grid(kv_dtype, C, S):
    # The last chunk of each row ends inside a tile (64 slots for 16-bit
    # caches, 128 for 8-bit ones), and so does the L2 prefetch of its first
    # tile (8, 40 or 72 slots here).  (1032, 16) plans 9 splits, past the
    # cluster merge, so the combine kernel runs; the others merge in
    # clusters.  Rows end at the capacity, one slot short of it, mid-row and
    # at slot 1, so some chunks start past their row's length.
    lens = [C, C - 1, C // 2 + 3, 1]
    w = inputs.custom(4, C, 1, kv_dtype=kv_dtype, kv_std=2.0 if kv_dtype == "e4m3" else 1.0, nan_tail=True)
    t = _make(w, lens=lens)
    p = _run(t, num_splits=S)
    assert gq.get_status(p) == 0
    _assert_parity(_gpu_rows(p.out), _oracle_full(t), f"{kv_dtype} C={C} S={S}")


def test_in_contract_lengths_raise_no_flags():
    t = _make(inputs.WORKLOADS[3])
    p = _run(t)
    assert gq.get_status(p) == 0


def test_errors_are_reported_before_launch():
    t = _make(inputs.custom(2, 128, 128))
    p = _prepare(t, num_splits=4)
    small = torch.zeros(256, dtype=torch.uint8, device=DEV)
    with pytest.raises(gq.GqaError) as e:
        api._lib.check(api._lib.load().gqa_decode_prepared(
            t["q"].data_ptr(), t["kv"].data_ptr(), t["lens"].data_ptr(), p.out.data_ptr(), 2, 128, 0,
            1.0, 4, small.data_ptr(), 256, None))
    assert e.value.name == "GQA_ERR_WORKSPACE_TOO_SMALL"
    with pytest.raises(ValueError):
        gq.prepare({"Q": t["q"], "KV": t["kv"], "O": t["q"], "sequence_lengths": t["lens"]})
    with pytest.raises(gq.GqaError) as e:
        api._lib.check(api._lib.load().gqa_decode_prepared(
            t["q"].data_ptr(), t["kv"].data_ptr(), t["lens"].data_ptr(), t["q"].data_ptr(), 2, 128, 0,
            1.0, 1, p.workspace.data_ptr(), p.workspace_bytes, None))
    assert e.value.name == "GQA_ERR_ALIASING"


@pytest.mark.parametrize("grid", ["cluster", "combine", "balanced"])
def test_stalled_pipeline_times_out_is_flagged_and_context_survives(grid):
    # The test hook never issues tile 3 of each split (of each CTA's stream
    # under the balanced schedule): the consumers' bounded wait runs out
    # after 100 ms, and so does the producer's wait for the stage they never
    # release; the CTAs flag GQA_FLAG_WAIT_TIMEOUT, skip their remaining
    # tiles, still pass every barrier of their epilogues (and, in a cluster,
    # the cluster barriers), drain their own copies and return.  No fault, no
    # hang; the next launch is fine.
    import time
    B, C, S = {"cluster": (1, 1024, 2),       # 16 CTAs of 8 tiles, clusters of 2
               "combine": (2, 4096, 16),      # one-wave grid of 256 CTAs of 4 tiles, 16 splits
               "balanced": (48, 2048, 8)}[grid]  # 3072 pieces > one wave: the balanced grid
    t = _make(inputs.custom(B, C, C))
    p = _prepare(t, num_splits=S)
    lib = api._lib.load()
    stream = torch.cuda.current_stream(DEV).cuda_stream
    t0 = time.time()
    st = lib.gqa_decode_debug_skip_tile(
        t["q"].data_ptr(), 0, t["kv"].data_ptr(), 0, t["lens"].data_ptr(), p.out.data_ptr(), B, C,
        1.0, 1.0, 1.0, S, p.workspace.data_ptr(), p.workspace_bytes, 3, 100_000_000, stream)
    assert st == 0, lib.gqa_last_error().decode()
    flags = gq.get_status(p)  # synchronises
    assert flags & api.FLAG_WAIT_TIMEOUT
    assert time.time() - t0 < 10.0
    gq.launch(p)
    torch.cuda.synchronize()
    assert gq.get_status(p) == 0
    _assert_parity(_gpu_rows(p.out), _oracle_full(t), "after a timed-out launch")



# ------------------------------------------------------------- paged cache


def _paged(pt, out=None, num_splits=None):
    w = pt["workload"]
    fp8 = w.kv_dtype == "e4m3"
    return gq.gqa_decode_paged(pt["q"], pt["kv_pages"], pt["block_table"], pt["lens"],
                               q_scale=pt["q_scale"], k_scale=pt["k_scale"] if fp8 else 1.0,
                               v_scale=pt["v_scale"] if fp8 else 1.0, out=out, num_splits=num_splits,
                               kv_scales=pt.get("kv_scale_pages"))


@pytest.mark.parametrize("q_dtype", ["bf16", "f16"])
@pytest.mark.parametrize("page_size", [16, 64, 256])
def test_paged_int8_matches_oracle_and_contiguous_path(q_dtype, page_size):
    # lengths with ragged scale tails (1, 17, 300: not multiples of 8) and
    # tiles spanning several 16-row pages
    w = inputs.custom(5, 1024, 1, 1024, kv_dtype="i8", q_dtype=q_dtype, nan_tail=True)
    t = _make(w, lens=[1, 17, 300, 1000, 1024])
    pt = inputs.paginate(t, page_size, extra_pages=5, seed=page_size)
    ref = _oracle_full(t)
    for S in (None, 3):
        out = _paged(pt, num_splits=S)
        torch.cuda.synchronize()
        _assert_parity(_gpu_rows(out), ref, f"paged int8 page {page_size} splits {S}")
        contiguous = _run(t, num_splits=S).out
        assert torch.equal(out.view(torch.int16), contiguous.view(torch.int16))


def test_paged_int8_balanced_schedule():
    rng = np.random.default_rng(12)
    C = 4096
    w = inputs.custom(48, C, 1, kv_dtype="i8", nan_tail=True)
    t = _make(w, lens=rng.integers(1, C + 1, 48).tolist())
    ref = _oracle_full(t)
    pt = inputs.paginate(t, 64, extra_pages=5)
    out = _paged(pt, num_splits=8)
    torch.cuda.synchronize()
    _assert_parity(_gpu_rows(out), ref, "paged int8, balanced")


@pytest.mark.parametrize("kv_dtype", ["f16", "e4m3", "i8"])
@pytest.mark.parametrize("T", [2, 4])
def test_paged_verify_window(kv_dtype, T):
    w = inputs.custom(4, 1024, T, 1024, kv_dtype=kv_dtype, kv_std=2.0 if kv_dtype == "e4m3" else 1.0,
                      nan_tail=True, q_len=T)
    t = _make(w, lens=[T, 100, 777, 1024])
    pt = inputs.paginate(t, 64, extra_pages=3, seed=T)
    ref = _oracle_full(t)
    for S in (None, 5):
        out = _paged(pt, num_splits=S)
        torch.cuda.synchronize()
        _assert_parity(_gpu_rows(out), ref, f"paged window {T} {kv_dtype} splits {S}")
        contiguous = _verify(t, num_splits=S)
        assert torch.equal(out.view(torch.int16), contiguous.view(torch.int16))


@pytest.mark.parametrize("kv_dtype,T", [("bf16", 2), ("i8", 2), ("e4m3", 3)])
def test_paged_verify_window_balanced(kv_dtype, T):
    # a ragged paged batch well past one wave: the balanced schedule (4 waves
    # for a 16-bit cache, 1 for 8-bit) with a window, pages shuffled
    B, C = 64, 2048
    rng = np.random.default_rng(31 + T)
    w = inputs.custom(B, C, 1, kv_dtype=kv_dtype, kv_std=2.0 if kv_dtype == "e4m3" else 1.0, nan_tail=True,
                      q_len=T)
    t = _make(w, lens=rng.integers(T, C + 1, B).tolist())
    ref = _oracle_full(t)
    pt = inputs.paginate(t, 128, extra_pages=9, seed=T)
    out = _paged(pt, num_splits=4)
    torch.cuda.synchronize()
    _assert_parity(_gpu_rows(out), ref, f"paged window {T} {kv_dtype}, balanced")


@pytest.mark.parametrize("kv_dtype", ["f16", "bf16", "e4m3"])
@pytest.mark.parametrize("page_size", [16, 64, 256])
def test_paged_matches_oracle_and_contiguous_path(kv_dtype, page_size):
    w = inputs.custom(5, 1024, 1, 1024, kv_dtype=kv_dtype, kv_std=2.0 if kv_dtype == "e4m3" else 1.0,
                      nan_tail=True)
    t = _make(w, lens=[1, 17, 300, 1000, 1024])
    pt = inputs.paginate(t, page_size, extra_pages=5, seed=page_size)
    for S in (None, 3):
        out = _paged(pt, num_splits=S)
        torch.cuda.synchronize()
        contiguous = _run(t, num_splits=S).out
        assert torch.equal(out.view(torch.int16), contiguous.view(torch.int16))
        g = oracle.gather_pages(bits_of(pt["kv_pages"]), pt["block_table"].cpu().numpy(),
                                t["lens"].cpu().numpy())
        ref, _ = oracle.gqa_decode(bits_of(t["q"]), FMT[w.q_dtype], g, FMT[kv_dtype], t["lens"].cpu().numpy(),
                                   q_scale=t["q_scale"], k_scale=t["k_scale"], v_scale=t["v_scale"])
        _assert_parity(_gpu_rows(out), ref, f"paged {kv_dtype} page {page_size} splits {S}")


def test_paged_out_of_range_page_ids_are_clamped_and_flagged():
    t = _make(inputs.custom(2, 512, 512))
    pt = inputs.paginate(t, 64, extra_pages=2)
    pt["block_table"][1, 3] = pt["num_pages"] + 10  # a used entry points outside the pool
    B, C, S = 2, 512, 2
    ws = torch.zeros(gq.workspace_size(B, C, S), dtype=torch.uint8, device=DEV)
    _paged_out = gq.gqa_decode_paged(pt["q"], pt["kv_pages"], pt["block_table"], pt["lens"],
                                     num_splits=S, workspace=ws)
    flags = gq.get_status(ws)
    assert flags & api.FLAG_PAGE_CLAMPED and not flags & api.FLAG_WAIT_TIMEOUT
    pt["block_table"][1, 3] = -4
    gq.gqa_decode_paged(pt["q"], pt["kv_pages"], pt["block_table"], pt["lens"], num_splits=S, workspace=ws)
    assert gq.get_status(ws) & api.FLAG_PAGE_CLAMPED


def test_paged_full_size_matches_oracle_and_contiguous():
    # the paged cache runs its own balanced schedule (4 waves of pieces), so
    # its FP32 rounding order differs from the contiguous launch: compare
    # both against the oracle on sampled units and with each other at the bar
    w = inputs.WORKLOADS[4]
    t = _make(w)
    contiguous = _run(t).out.clone()
    rng = np.random.default_rng(44)
    units = sorted({(int(b), int(g)) for b, g in zip(rng.integers(0, w.batch, 4), rng.integers(0, 8, 4))}
                   | {(0, 0), (w.batch - 1, 7)})
    ref = _oracle_units(t, units)
    pt = inputs.paginate(t, 256, extra_pages=7)
    del t["kv"]
    out = _paged(pt)
    torch.cuda.synchronize()
    got = _gpu_rows(out)
    rows = sorted(ref)
    _assert_parity(got[rows], np.stack([ref[r] for r in rows]), "paged full size, sampled", rms_gate=True)
    _assert_parity(got, _gpu_rows(contiguous).astype(np.float64), "paged vs contiguous", rms_gate=True)



# ----------------------------------------------------------- verify window


def test_workspace_init_zeroes_a_dirty_workspace():
    t = _make(inputs.custom(5, 2048, 1, 2048, kv_dtype="bf16"))
    S = 8
    ws = torch.full((gq.workspace_size(5, 2048, S),), 0xA5, dtype=torch.uint8, device=DEV)
    gq.workspace_init(ws)
    assert int(ws[:256].sum()) == 0
    p = _prepare(t, num_splits=S, workspace=ws)
    gq.launch(p)
    torch.cuda.synchronize()
    assert gq.get_status(p) == 0
    _assert_parity(_gpu_rows(p.out), _oracle_full(t), "after workspace_init")


def _verify(t, num_splits=None):
    w = t["workload"]
    fp8 = w.kv_dtype == "e4m3"
    q = t["q"] if t["q"].dim() == 4 else t["q"][:, None].contiguous()  # [B, T, 32, 128]
    out = gq.gqa_decode_verify(q, t["kv"], t["lens"], q_scale=t["q_scale"],
                               k_scale=t["k_scale"] if fp8 else 1.0, v_scale=t["v_scale"] if fp8 else 1.0,
                               kv_scales=t["kv_scales"], num_splits=num_splits)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("kv_dtype", ["f16", "bf16", "e4m3", "i8"])
@pytest.mark.parametrize("T", [1, 2, 3, 4])
def test_verify_window_every_element(kv_dtype, T):
    w = inputs.custom(6, 1024, T, 1024, kv_dtype=kv_dtype, kv_std=2.0 if kv_dtype == "e4m3" else 1.0,
                      nan_tail=True, q_len=T)
    t = _make(w, lens=[T, T + 1, 63 + T, 64, 500, 1024])
    for S in (None, 1, 3):
        out = _verify(t, num_splits=S)
        _assert_parity(_gpu_rows(out), _oracle_full(t), f"verify T={T} {kv_dtype} splits={S}")


@pytest.mark.parametrize("kv_dtype,T", [("f16", 1), ("bf16", 1), ("e4m3", 1), ("i8", 1), ("bf16", 3)])
def test_cluster_merge_every_split_count(kv_dtype, T):
    # one-piece grids of 2..8 splits run as one thread-block cluster per
    # (row, KV head) and merge on chip; row 0 holds slots in its first split
    # only, so the other members of its clusters merge empty states.  16
    # splits (16-bit KV; 2048 slots give 8-bit KV at most 8) merge through
    # the combine kernel instead: the control.
    C = 2048
    w = inputs.custom(3, C, T, kv_dtype=kv_dtype, kv_std=2.0 if kv_dtype == "e4m3" else 1.0, nan_tail=True,
                      q_len=T)
    t = _make(w, lens=[T, 700, C])
    ref = _oracle_full(t)
    for S in list(range(2, 9)) + [16]:
        out = _verify(t, num_splits=S) if T > 1 else _run(t, num_splits=S).out
        _assert_parity(_gpu_rows(out), ref, f"{kv_dtype} T={T} splits={S}")


@pytest.mark.parametrize("B,T,merged_on_chip", [(2, 1, True), (2, 2, True), (64, 2, False)])
def test_cluster_merge_only_for_single_wave_grids(B, T, merged_on_chip):
    # the cluster merge writes no partials: a workspace whose partial area
    # holds a sentinel keeps it when the 4 splits merge on chip (a one-wave
    # grid: 8 x 2 x 4 CTAs) and loses it when the combine kernel merges
    # (8 x 64 x 4 = 2048 CTAs, several waves).  Both match the oracle.
    C, S = 1024, 4
    t = _make(inputs.custom(B, C, C, q_len=T))
    ws = torch.full((gq.workspace_size(B * T, C, S),), 0xA5, dtype=torch.uint8, device=DEV)
    gq.workspace_init(ws)
    if T == 1:
        p = _prepare(t, num_splits=S, workspace=ws)
        gq.launch(p)
        out = p.out
    else:
        out = gq.gqa_decode_verify(t["q"], t["kv"], t["lens"], num_splits=S, workspace=ws)
    torch.cuda.synchronize()
    untouched = bool(torch.all(ws[256:] == 0xA5))
    assert untouched == merged_on_chip
    _assert_parity(_gpu_rows(out), _oracle_full(t), f"B={B} T={T} splits={S}")


@pytest.mark.parametrize("kv_dtype,B,S", [("e4m3", 8, 7), ("e4m3", 8, 6), ("i8", 8, 7), ("bf16", 4, 8),
                                           ("bf16", 8, 4), ("f16", 19, 2)])
def test_cluster_merge_matches_the_launch_count(kv_dtype, B, S):
    # one-wave grids near full occupancy: the merge stays on chip only when
    # every cluster can be resident at once (the device's cluster occupancy),
    # else the combine kernel merges; the host-side launch count says which,
    # the partial area shows which ran, and both match the oracle
    C = 4096
    w = inputs.custom(B, C, C // 2, C, kv_dtype=kv_dtype, kv_std=2.0 if kv_dtype == "e4m3" else 1.0)
    t = _make(w)
    fp8 = kv_dtype == "e4m3"
    ws = torch.full((gq.workspace_size(B, C, S),), 0xA5, dtype=torch.uint8, device=DEV)
    gq.workspace_init(ws)
    p = _prepare(t, num_splits=S, workspace=ws)
    gq.launch(p)
    torch.cuda.synchronize()
    kvf = {"f16": api.KV_F16, "bf16": api.KV_BF16, "e4m3": api.KV_E4M3, "i8": api.KV_I8}[kv_dtype]
    n = api.launch_count(B, C, kvf, 1, S, torch.cuda.get_device_properties(DEV).multi_processor_count)
    on_chip = bool(torch.all(ws[256:] == 0xA5))
    print(f"PARITY cluster {kv_dtype} B={B} S={S}: {'on chip' if on_chip else 'combine kernel'}")
    assert on_chip == (n == 1)
    _assert_parity(_gpu_rows(p.out), _oracle_full(t), f"{kv_dtype} B={B} splits={S}")


@pytest.mark.parametrize("kv_dtype", ["f16", "bf16", "e4m3", "i8"])
@pytest.mark.parametrize("T", [2, 4])
def test_balanced_verify_window(kv_dtype, T):
    # a ragged batch well past one wave runs the balanced schedule with a
    # window too: rows are cut at run ends, and a piece may hold no slot for
    # an early query of the window (its causal limit); lengths below T give
    # zero rows for the queries without slots and the clamp flag
    B, C = 96, 2048
    rng = np.random.default_rng(T)
    lens = rng.integers(T, C + 1, B)
    lens[:6] = [T - 1, T, T + 1, 64, C, C - 1]
    w = inputs.custom(B, C, 1, kv_dtype=kv_dtype, kv_std=2.0 if kv_dtype == "e4m3" else 1.0, nan_tail=True,
                      q_len=T)
    t = _make(w, lens=lens.tolist())
    fp8 = kv_dtype == "e4m3"
    ws = torch.zeros(gq.workspace_size(B * T, C, 4), dtype=torch.uint8, device=DEV)
    out = gq.gqa_decode_verify(t["q"], t["kv"], t["lens"], q_scale=t["q_scale"],
                               k_scale=t["k_scale"] if fp8 else 1.0, v_scale=t["v_scale"] if fp8 else 1.0,
                               kv_scales=t["kv_scales"], num_splits=4, workspace=ws)
    assert gq.get_status(ws) & api.FLAG_LENGTH_CLAMPED
    got = out.view(B, T, 32, 128)
    assert not got[0, 0].any()  # length T - 1: the first query has no slot
    keep = list(range(1, B))
    sub = dict(t, q=t["q"][keep], kv=t["kv"][keep], lens=t["lens"][keep],
               kv_scales=t["kv_scales"][keep] if t["kv_scales"] is not None else None)
    _assert_parity(_gpu_rows(got[keep]), _oracle_full(sub), f"balanced window T={T} {kv_dtype}")


def test_verify_window_of_one_is_the_plain_decode():
    t = _make(inputs.WORKLOADS[3])
    plain = _run(t).out
    t1 = dict(t, q=t["q"][:, None].contiguous())
    out = _verify(t1)
    assert torch.equal(out[:, 0].contiguous().view(torch.int16), plain.view(torch.int16))


def test_verify_window_lengths_below_q_len_give_zero_rows_and_a_flag():
    T, C = 3, 256
    t = _make(inputs.custom(2, C, 2, 2, q_len=T), lens=[2, 200])  # row 0: only queries 1, 2 have slots
    ws = torch.zeros(gq.workspace_size(2 * T, C, 4), dtype=torch.uint8, device=DEV)
    out = gq.gqa_decode_verify(t["q"], t["kv"], t["lens"], num_splits=4, workspace=ws)
    assert gq.get_status(ws) & api.FLAG_LENGTH_CLAMPED
    assert torch.all(out[0, 0] == 0)
    ref = oracle.gqa_decode(bits_of(t["q"][1:]), oracle.F16, bits_of(t["kv"][1:]), oracle.F16,
                            np.array([200], np.int32))[0]
    _assert_parity(_gpu_rows(out[1:]), ref, "verify row with a valid length")


def test_verify_window_medium_size_bf16():
    t = _make(inputs.custom(4, 16384, 8000, 16384, kv_dtype="bf16", q_len=2))
    out = _verify(t)
    _assert_parity(_gpu_rows(out), _oracle_full(t), "verify T=2 bf16 4 x U[8000,16384]")



# --------------------------------------------------- K/V append (before decode)


def _append_inputs(B, C, dtype, seed=0):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    dt = {"f16": torch.float16, "bf16": torch.bfloat16}[dtype]
    rnd = lambda *shape: torch.randn(shape, generator=g, device=DEV, dtype=torch.float32)  # noqa: E731
    qp, kp, vp = rnd(B, 32, 128).to(dt), rnd(B, 8, 128).to(dt), rnd(B, 8, 128).to(dt)
    wq, wk = (1 + 0.1 * rnd(128)).to(dt), (1 + 0.1 * rnd(128)).to(dt)
    pos = torch.randint(0, 200000, (B,), generator=g, device=DEV, dtype=torch.int32)
    slots = torch.randint(0, C, (B,), generator=g, device=DEV, dtype=torch.int32)
    return qp, kp, vp, wq, wk, pos, slots


def _vals(t):
    return t.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_append_matches_oracle_and_touches_only_its_slot(dtype):
    # An element-wise step rounded once: every q_out and K element must be the
    # oracle's correctly rounded value or one of its two neighbours (the kernel
    # rounds an FP32 value within ~2^-21 of exact; the oracle an FP64 one).
    B, C = 6, 300
    qp, kp, vp, wq, wk, pos, slots = _append_inputs(B, C, dtype, seed=1)
    kv = _make(inputs.custom(B, C, C, kv_dtype=dtype))["kv"]
    before = kv.clone()
    q_out = gq.append_kv(qp, kp, vp, wq, wk, pos, slots, kv, eps=1e-6, rope_theta=1e6)
    torch.cuda.synchronize()
    qo, ko, vo = oracle.append_kv(_vals(qp), _vals(kp), _vals(vp), _vals(wq), _vals(wk),
                                  pos.cpu().numpy(), 1e-6, 1e6)
    fmt = FMT[dtype]
    d_q = ulps_apart(bits_of(q_out), oracle.round_to(qo, fmt))
    assert d_q.max() <= 1, f"append q_out {dtype}: {int(d_q.max())} ulps from the oracle"
    sl = slots.cpu().tolist()
    k_new = torch.stack([kv[b, 0, :, sl[b]] for b in range(B)])
    d_k = ulps_apart(bits_of(k_new), oracle.round_to(ko, fmt))
    assert d_k.max() <= 1, f"append k {dtype}: {int(d_k.max())} ulps from the oracle"
    print(f"PARITY append {dtype}: q_out {np.mean(d_q > 0):.2%}, k {np.mean(d_k > 0):.2%} of elements one ulp off")
    v_new = torch.stack([kv[b, 1, :, sl[b]] for b in range(B)])
    assert torch.equal(v_new.view(torch.int16), vp.view(torch.int16))
    for b in range(B):  # nothing else in the cache changed
        before[b, :, :, sl[b]] = kv[b, :, :, sl[b]]
    assert torch.equal(kv.view(torch.int16), before.view(torch.int16))


@pytest.mark.parametrize("theta", [1e4, 1e6])
def test_append_rotary_angles_up_to_2_31(theta):
    # The kernel takes the rotary sine and cosine by its own reduction modulo
    # pi/2 and Taylor series: positions up to 2^31 - 1 (angles up to 2^31
    # radians for the first frequency), each still within one ulp of the
    # oracle's RNE value for every q_out and K element.
    positions = [0, 1, 2 ** 20, 2 ** 24 + 1, 2 ** 30, 2 ** 31 - 1]
    B, C = len(positions), 64
    qp, kp, vp, wq, wk, _, slots = _append_inputs(B, C, "bf16", seed=21)
    pos = torch.tensor(positions, dtype=torch.int32, device=DEV)
    kv = _make(inputs.custom(B, C, C, kv_dtype="bf16"))["kv"]
    q_out = gq.append_kv(qp, kp, vp, wq, wk, pos, slots, kv, eps=1e-6, rope_theta=theta)
    torch.cuda.synchronize()
    qo, ko, _ = oracle.append_kv(_vals(qp), _vals(kp), _vals(vp), _vals(wq), _vals(wk), pos.cpu().numpy(), 1e-6,
                                 theta)
    d_q = ulps_apart(bits_of(q_out), oracle.round_to(qo, FMT["bf16"]))
    sl = slots.cpu().tolist()
    k_new = torch.stack([kv[b, 0, :, sl[b]] for b in range(B)])
    d_k = ulps_apart(bits_of(k_new), oracle.round_to(ko, FMT["bf16"]))
    assert d_q.max() <= 1 and d_k.max() <= 1, f"theta {theta}: q {int(d_q.max())}, k {int(d_k.max())} ulps"


def _nearest_codes(ref, table_vals):
    """Indices of the two representable values bracketing ref (sorted table)."""
    i = np.searchsorted(table_vals, ref)
    return np.clip(i - 1, 0, len(table_vals) - 1), np.clip(i, 0, len(table_vals) - 1)


@pytest.mark.parametrize("fmt", ["e4m3", "i8"])
def test_append_quantising_writes(fmt):
    B, C = 4, 256
    qp, kp, vp, wq, wk, pos, slots = _append_inputs(B, C, "bf16", seed=2)
    w = inputs.custom(B, C, C, kv_dtype=fmt, kv_std=2.0 if fmt == "e4m3" else 1.0)
    t = _make(w)
    kv, sc = t["kv"], t["kv_scales"]
    ks, vs = (0.02, 0.03) if fmt == "e4m3" else (1.0, 1.0)
    gq.append_kv(qp, kp, vp, wq, wk, pos, slots, kv, k_scale=ks, v_scale=vs, kv_scales=sc)
    torch.cuda.synchronize()
    _, ko, vo = oracle.append_kv(_vals(qp), _vals(kp), _vals(vp), _vals(wq), _vals(wk), pos.cpu().numpy(),
                                 1e-6, 1e6)
    sl = slots.cpu().tolist()
    for b in range(B):
        for plane, ref_rows, scale in ((0, ko[b], ks), (1, vo[b], vs)):
            codes = kv[b, plane, :, sl[b]].cpu()
            if fmt == "e4m3":
                got = torch.from_numpy(codes.numpy()).view(torch.float8_e4m3fn).double().numpy()
                ref = ref_rows / scale
                # the kernel's choice must be one of the two e4m3 values bracketing ref
                table = np.sort(np.unique(torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn)
                                          .double().numpy()))
                table = table[np.isfinite(table)]
                lo, hi = _nearest_codes(ref, table)
                ok = (got == table[lo]) | (got == table[hi])
                assert ok.all(), f"e4m3 codes off the bracketing pair at b={b} plane={plane}"
            else:
                row_scale = sc[b, plane, :, sl[b]].double().cpu().numpy()  # [8]
                amax = np.abs(ref_rows).max(axis=1)
                np.testing.assert_allclose(row_scale, amax / 127, rtol=2 ** -7)  # bf16 of amax/127
                got = codes.numpy().astype(np.float64) * row_scale[:, None]
                assert np.all(np.abs(got - ref_rows) <= 0.5 * row_scale[:, None] * (1 + 1e-3) + 1e-6)


def test_append_out_of_range_slot_is_skipped_and_flagged():
    B, C = 3, 128
    qp, kp, vp, wq, wk, pos, _ = _append_inputs(B, C, "bf16", seed=3)
    slots = torch.tensor([5, C + 3, -1], dtype=torch.int32, device=DEV)
    kv = _make(inputs.custom(B, C, C, kv_dtype="bf16"))["kv"]
    before = kv.clone()
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    gq.append_kv(qp, kp, vp, wq, wk, pos, slots, kv, workspace=ws)
    assert gq.get_status(ws) & api.FLAG_SLOT_CLAMPED
    before[0, :, :, 5] = kv[0, :, :, 5]
    assert torch.equal(kv.view(torch.int16), before.view(torch.int16))


def _append_fmt_inputs(fmt, B, C, seed):
    dtype = "bf16" if fmt in ("bf16", "e4m3", "i8") else "f16"
    qp, kp, vp, wq, wk, pos, _ = _append_inputs(B, C, dtype, seed=seed)
    return dtype, qp, kp, vp, wq, wk, pos


@pytest.mark.parametrize("fmt", ["f16", "bf16", "e4m3", "i8"])
@pytest.mark.parametrize("page_size", [16, 64])
def test_append_paged_equals_contiguous(fmt, page_size):
    # the same token appended into a paged cache and into the contiguous cache
    # it was paged from: the pool gathered back equals the contiguous cache bit
    # for bit, and the decodes that follow agree bit for bit
    B, C = 4, 1024
    lens = [page_size * k + 5 for k in (1, 3, 7, 11)]  # the next slot stays in a used page
    w = inputs.custom(B, C, 1, kv_dtype=fmt, q_dtype="bf16" if fmt in ("e4m3", "i8") else fmt,
                      kv_std=2.0 if fmt == "e4m3" else 1.0)
    t = _make(w, lens=lens)
    pt = inputs.paginate(t, page_size, extra_pages=3, seed=page_size)
    _, qp, kp, vp, wq, wk, pos = _append_fmt_inputs(fmt, B, C, seed=13)
    slots = t["lens"].clone()
    ks = t["k_scale"] if fmt == "e4m3" else 1.0
    vs = t["v_scale"] if fmt == "e4m3" else 1.0
    q1 = gq.append_kv(qp, kp, vp, wq, wk, pos, slots, t["kv"], k_scale=ks, v_scale=vs,
                      kv_scales=t["kv_scales"])
    q2 = gq.append_kv_paged(qp, kp, vp, wq, wk, pos, slots, pt["kv_pages"], pt["block_table"], k_scale=ks,
                            v_scale=vs, kv_scales=pt.get("kv_scale_pages"))
    torch.cuda.synchronize()
    assert torch.equal(q1.view(torch.int16), q2.view(torch.int16))
    lens1 = (slots + 1).cpu().numpy()
    g = oracle.gather_pages(bits_of(pt["kv_pages"]), pt["block_table"].cpu().numpy(), lens1)
    kvb = bits_of(t["kv"])
    for b in range(B):
        assert np.array_equal(g[b, :, :, :lens1[b]], kvb[b, :, :, :lens1[b]])
    if fmt == "i8":
        gs = oracle.gather_pages(bits_of(pt["kv_scale_pages"]), pt["block_table"].cpu().numpy(), lens1)
        sb = bits_of(t["kv_scales"])
        for b in range(B):
            assert np.array_equal(gs[b, :, :, :lens1[b]], sb[b, :, :, :lens1[b]])
    t["lens"].copy_(slots + 1)
    t["q"] = q1
    pt["q"] = q2
    out_c = _run(t, num_splits=4).out
    out_p = _paged(pt, num_splits=4)
    torch.cuda.synchronize()
    assert torch.equal(out_c.view(torch.int16), out_p.view(torch.int16))


def test_append_paged_out_of_range_entry_is_not_written():
    B, C, ps = 2, 512, 64
    t = _make(inputs.custom(B, C, 100, 100))
    pt = inputs.paginate(t, ps, extra_pages=1)
    _, qp, kp, vp, wq, wk, pos = _append_fmt_inputs("f16", B, C, seed=14)
    slots = torch.tensor([100, 101], dtype=torch.int32, device=DEV)
    pt["block_table"][0, 100 // ps] = pt["num_pages"] + 3  # row 0's page for its slot is out of range
    before = pt["kv_pages"].clone()
    hdr = torch.zeros(256, dtype=torch.uint8, device=DEV)
    q_out = gq.append_kv_paged(qp, kp, vp, wq, wk, pos, slots, pt["kv_pages"], pt["block_table"], workspace=hdr)
    torch.cuda.synchronize()
    assert gq.get_status(hdr) & api.FLAG_PAGE_CLAMPED
    page1 = int(pt["block_table"][1, 101 // ps])
    changed = (pt["kv_pages"].view(torch.int16) != before.view(torch.int16)).flatten(1).any(1)  # per page, bits
    assert changed.nonzero().flatten().tolist() == [page1]  # only row 1's page was written
    assert torch.isfinite(q_out.float()).all()


def test_append_then_decode_matches_the_oracle_chain():
    # GPU: append the new token, then decode over len = slot + 1.  Oracle: the
    # same two steps computed from the same inputs, rounding the appended rows
    # with its own RNE, never reading anything the GPU produced.
    B, C = 4, 2048
    qp, kp, vp, wq, wk, pos, _ = _append_inputs(B, C, "bf16", seed=4)
    t = _make(inputs.custom(B, C, 1000, 2000, kv_dtype="bf16"))
    slots = t["lens"].clone()                       # append at the current length
    kv_bits0 = bits_of(t["kv"]).copy()
    q_out = gq.append_kv(qp, kp, vp, wq, wk, pos, slots, t["kv"])
    lens = slots + 1
    out = gq.gqa_decode(q_out, t["kv"], lens)
    torch.cuda.synchronize()
    qo, ko, vo = oracle.append_kv(_vals(qp), _vals(kp), _vals(vp), _vals(wq), _vals(wk), pos.cpu().numpy(),
                                  1e-6, 1e6)
    q_bits = oracle.round_to(qo, oracle.BF16)
    for b, s_ in enumerate(slots.cpu().tolist()):
        kv_bits0[b, 0, :, s_] = oracle.round_to(ko[b], oracle.BF16)
        kv_bits0[b, 1, :, s_] = bits_of(vp[b])
    ref, _ = oracle.gqa_decode(q_bits, oracle.BF16, kv_bits0, oracle.BF16, lens.cpu().numpy())
    _assert_parity(_gpu_rows(out), ref, "append -> decode chain")


# ------------------------------------------------ CUDA graphs beyond prepare


def _replay_equals_eager(step, outs):
    """Capture `step` (no allocation, no host sync inside), replay it, and
    compare with an eager run on the same inputs, bit for bit."""
    step()
    torch.cuda.synchronize()
    eager = [o.clone() for o in outs]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # warm-up on a side stream before capture
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for o in outs:
        o.zero_()
    g.replay()
    torch.cuda.synchronize()
    for o, e in zip(outs, eager):
        assert torch.equal(o.view(torch.int16) if o.element_size() == 2 else o, e.view(torch.int16)
                           if e.element_size() == 2 else e)
    return g


def test_graph_append_then_decode_serving_step():
    # one decode step of a server as one graph: append the new token (norm,
    # RoPE, cache write at `slots`), then decode over len = slot + 1; the
    # next step only rewrites inputs in place and replays
    B, C = 8, 4096
    qp, kp, vp, wq, wk, pos, _ = _append_inputs(B, C, "bf16", seed=9)
    t = _make(inputs.custom(B, C, 1000, 3000, kv_dtype="bf16"))
    slots = t["lens"].clone()
    lens = slots + 1
    q_out = torch.empty_like(qp)
    out = torch.empty_like(qp)
    hdr = torch.zeros(256, dtype=torch.uint8, device=DEV)
    S = 8
    p = gq.prepare({"Q": q_out, "KV": t["kv"], "O": out, "sequence_lengths": lens}, num_splits=S)

    def step():
        gq.append_kv(qp, kp, vp, wq, wk, pos, slots, t["kv"], q_out=q_out, workspace=hdr)
        gq.launch(p)

    g = _replay_equals_eager(step, [q_out, out])
    # next token: new projections, positions, slots and lengths written in place
    qp2, kp2, vp2, _, _, _, _ = _append_inputs(B, C, "bf16", seed=10)
    kv_before = t["kv"].clone()
    for dst, src in ((qp, qp2), (kp, kp2), (vp, vp2)):
        dst.copy_(src)
    pos.add_(1)
    slots.add_(1)
    lens.add_(1)
    g.replay()
    torch.cuda.synchronize()
    replayed = out.clone()
    t["kv"].copy_(kv_before)
    step()
    torch.cuda.synchronize()
    assert torch.equal(replayed.view(torch.int16), out.view(torch.int16))
    assert gq.get_status(hdr) == 0


@pytest.mark.parametrize("kind", ["paged", "int8", "verify2"])
def test_graph_capture_other_entry_points(kind):
    B, C, S = 16, 2048, 8
    rng = np.random.default_rng(21)
    lens = rng.integers(1, C + 1, B).tolist()
    if kind == "int8":
        t = _make(inputs.custom(B, C, 1, kv_dtype="i8"), lens=lens)
    elif kind == "verify2":
        t = _make(inputs.custom(B, C, 2, q_len=2), lens=[max(2, x) for x in lens])
    else:
        t = _make(inputs.custom(B, C, 1), lens=lens)
    out = torch.empty_like(t["q"])
    rows = B * (2 if kind == "verify2" else 1)
    ws = torch.zeros(gq.workspace_size(rows, C, S), dtype=torch.uint8, device=DEV)
    if kind == "paged":
        pt = inputs.paginate(t, 64, extra_pages=3)

        def step():
            gq.gqa_decode_paged(pt["q"], pt["kv_pages"], pt["block_table"], pt["lens"], out=out,
                                num_splits=S, workspace=ws)
    elif kind == "int8":
        def step():
            gq.gqa_decode_int8kv(t["q"], t["kv"], t["kv_scales"], t["lens"], out=out, num_splits=S,
                                 workspace=ws)
    else:
        def step():
            gq.gqa_decode_verify(t["q"], t["kv"], t["lens"], out=out, num_splits=S, workspace=ws)
    g = _replay_equals_eager(step, [out])
    _assert_parity(_gpu_rows(out), _oracle_full(t), f"graph {kind}")
    # shorter lengths, written in place, then replay
    lens_t = pt["lens"] if kind == "paged" else t["lens"]
    lens_t.copy_(torch.clamp(lens_t // 2, min=2))
    g.replay()
    torch.cuda.synchronize()
    if kind == "paged":
        t["lens"] = pt["lens"]
    _assert_parity(_gpu_rows(out), _oracle_full(t), f"graph {kind}, lengths halved")
