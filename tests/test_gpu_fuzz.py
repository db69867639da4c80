"""Seeded random cases through the C ABI against the FP64 oracle, every element.

The fixed-shape parity tests pin chosen edge cases; these draw the rest at
random so that the launch paths meet in combinations nobody picked: the KV
format (fp16, bf16, e4m3, int8 with row scales), the window (1-4 query
tokens), batch and capacity, uniform or ragged lengths (some rows empty),
the split count (planner or explicit), and a contiguous or paged cache
(shuffled pages of 16-256 slots).  With an 8-bit cache, q's magnitude is
drawn from 1e-7 to 1e6 as well (q_scale compensates).  Together they reach every schedule: one
piece per CTA merged by the combine kernel, one-wave grids merged on chip in
thread-block clusters, and the balanced schedule with and without the
per-row cost, single tokens and windows, 1 or 4 waves.  Sizes stay small
enough for the oracle to check every output element in a few seconds.
"""
import numpy as np
import pytest
import torch

import oracle
import gqa_decode_attention_sm_gb300 as gq
from gqa_decode_attention_sm_gb300 import inputs
from helpers import bits_of, tolerance_ok, ulps_apart

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
FMT = {"f16": oracle.F16, "bf16": oracle.BF16, "e4m3": oracle.E4M3, "i8": oracle.I8}
N_CASES = 48


def _cases():
    rng = np.random.default_rng(2026)
    out = []
    while len(out) < N_CASES:
        kv_dtype = str(rng.choice(["f16", "bf16", "e4m3", "i8"]))
        T = int(rng.choice([1, 1, 1, 2, 3, 4]))
        paged = bool(rng.random() < 0.4)
        page = int(rng.choice([16, 64, 256]))
        B = int(rng.choice([1, 2, 3, 5, 8, 17, 40, 96, 160]))
        C = int(rng.choice([64, 128, 256, 512, 768, 1024, 2048]))
        if paged:
            C = max(page, C // page * page)
        if B * C * T > 400_000:
            continue
        kind = str(rng.choice(["uniform", "ragged", "ragged", "ragged_empty"]))
        if kind == "uniform":
            lens = [C] * B
        else:
            lens = rng.integers(T, C + 1, B).tolist()
            if kind == "ragged_empty" and B > 1:
                for b in rng.choice(B, size=max(1, B // 8), replace=False):
                    lens[int(b)] = 0
        S = rng.choice([None, None, None, 1, 2, 3, 4, 8, 16, 38])
        S = None if S is None else int(S)
        q_scale = float(rng.choice([1.0, 0.5, 2.0]))
        out.append((len(out), kv_dtype, T, paged, page, B, C, [int(x) for x in lens], S, q_scale))
    return out


def _balanced_cases():
    """Cases built to need the balanced schedule: batches of 48-128 rows,
    capacity >= 1024 and 4-16 splits put the one-piece grid past one wave."""
    rng = np.random.default_rng(7)
    out = []
    while len(out) < 16:
        kv_dtype = str(rng.choice(["f16", "bf16", "e4m3", "i8"]))
        T = int(rng.choice([1, 1, 2, 3, 4]))
        paged = bool(rng.random() < 0.4)
        page = int(rng.choice([64, 256]))
        B = int(rng.choice([48, 64, 96, 128]))
        C = int(rng.choice([1024, 2048]))
        if B * C * T > 400_000:
            continue
        lens = rng.integers(T, C + 1, B).tolist()
        if rng.random() < 0.3:
            for b in rng.choice(B, size=B // 10, replace=False):
                lens[int(b)] = 0
        if rng.random() < 0.2:
            lens = [C] * B
        S = int(rng.choice([4, 8, 16]))
        q_scale = float(rng.choice([1.0, 0.5, 2.0]))
        out.append((100 + len(out), kv_dtype, T, paged, page, B, C, [int(x) for x in lens], S, q_scale))
    return out


def _long_row_cases():
    """Automatic plans for batches of 8-16 rows of 4096-8192 slots, where
    the one-wave grid gives way to the balanced schedule; uniform and ragged
    lengths, 1-2 query tokens, contiguous or paged."""
    rng = np.random.default_rng(11)
    out = []
    while len(out) < 8:
        kv_dtype = str(rng.choice(["f16", "bf16", "e4m3", "i8"]))
        T = int(rng.choice([1, 1, 2]))
        B = int(rng.choice([8, 12, 16]))
        C = int(rng.choice([4096, 6144, 8192]))
        if B * C * T > 140_000:
            continue
        paged = bool(rng.random() < 0.3)
        lens = [C] * B if rng.random() < 0.3 else rng.integers(max(T, C // 4), C + 1, B).tolist()
        out.append((200 + len(out), kv_dtype, T, paged, 256, B, C, [int(x) for x in lens], None, 1.0))
    return out


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gqa_decode_attention_sm_gb300 import build as gbuild
    gbuild.build()
    oracle.build()
    torch.cuda.init()


@pytest.mark.parametrize("case", _cases() + _balanced_cases() + _long_row_cases(), ids=lambda c: f"case{c[0]}-{c[1]}-T{c[2]}-{'paged' if c[3] else 'contig'}"
                         f"-B{c[5]}-C{c[6]}-S{c[8]}")
def test_random_case_matches_oracle(case):
    idx, kv_dtype, T, paged, page, B, C, lens, S, q_scale = case
    fp8 = kv_dtype == "e4m3"
    w = inputs.custom(B, C, 1, kv_dtype=kv_dtype, kv_std=2.0 if fp8 else 1.0, nan_tail=True, q_scale=q_scale,
                      index=500 + idx, q_len=T)
    t = inputs.make(w, DEV, lens=lens)
    if kv_dtype in ("e4m3", "i8"):
        # 8-bit caches run f16 tensor cores on a bf16 q: draw q's magnitude
        # from 1e-7 to 1e6 (q_scale divided by the same factor keeps the
        # softmax ordinary), so every case also crosses the f16 range that
        # the per-column power-of-two scaling bridges
        f = float(10.0 ** np.random.default_rng(9000 + idx).uniform(-7.0, 6.0))
        t["q"] = (t["q"].float() * f).to(t["q"].dtype)
        q_scale = q_scale / f
    ks, vs = (t["k_scale"], t["v_scale"]) if fp8 else (1.0, 1.0)
    q4 = t["q"] if T > 1 else t["q"][:, None].contiguous()
    if paged:
        pt = inputs.paginate(t, page, extra_pages=3, seed=idx)
        out = gq.gqa_decode_paged(q4 if T > 1 else t["q"], pt["kv_pages"], pt["block_table"], pt["lens"],
                                  q_scale=q_scale, k_scale=ks, v_scale=vs, num_splits=S,
                                  kv_scales=pt.get("kv_scale_pages"))
    else:
        out = gq.gqa_decode_verify(q4, t["kv"], t["lens"], q_scale=q_scale, k_scale=ks, v_scale=vs,
                                   kv_scales=t["kv_scales"], num_splits=S)
    torch.cuda.synchronize()
    got = out.float().view(B, T, 32, 128).cpu().numpy()
    keep = [b for b in range(B) if lens[b] > 0]
    empty = [b for b in range(B) if lens[b] == 0]
    assert not np.any(got[empty]), "rows without slots must be zero"
    if not keep:
        return
    args = dict(q_scale=q_scale, k_scale=t["k_scale"], v_scale=t["v_scale"])
    if t["kv_scales"] is not None:
        args["kv_scales"] = bits_of(t["kv_scales"][keep])
    qk = t["q"][keep]
    ref, _ = oracle.gqa_decode(bits_of(qk), FMT[w.q_dtype], bits_of(t["kv"][keep]), FMT[kv_dtype],
                               np.array([lens[b] for b in keep], np.int32), **args)
    ok, err, excess = tolerance_ok(got[keep].reshape(-1, 128), ref)
    assert ok, f"case {idx}: max |gpu - oracle| {err:.3e} exceeds the bar by {excess:.3e}"


# ------------------------------------------------------- the append step


def _append_cases():
    """Seeded random append steps: cache format and projection dtype, batch,
    capacity, contiguous or paged (16- or 64-slot pages), rotary positions
    up to 2^21, input magnitudes from 1e-3 to 1e3 (the RMS norm must undo
    them; at 1e-3 eps matters), eps and theta."""
    rng = np.random.default_rng(4242)
    out = []
    for idx in range(24):
        fmt = str(rng.choice(["f16", "bf16", "e4m3", "i8"]))
        dtype = fmt if fmt in ("f16", "bf16") else str(rng.choice(["f16", "bf16"]))
        B = int(rng.choice([1, 2, 5, 16, 33, 64]))
        C = int(rng.choice([64, 256, 1024]))
        paged = bool(rng.random() < 0.5)
        page = int(rng.choice([16, 64]))
        pos_hi = int(rng.choice([16, 4096, 1 << 21]))
        mag = float(10.0 ** rng.uniform(-3.0, 3.0))
        eps = float(rng.choice([1e-6, 1e-5]))
        theta = float(rng.choice([1e4, 5e5, 1e6]))
        out.append((idx, fmt, dtype, B, C, paged, page, pos_hi, mag, eps, theta))
    return out


def _e4m3_table():
    t = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    return np.sort(np.unique(t[np.isfinite(t)]))


@pytest.mark.parametrize("case", _append_cases(),
                         ids=lambda c: f"append{c[0]}-{c[1]}-{c[2]}-B{c[3]}-C{c[4]}-{'paged' if c[5] else 'contig'}")
def test_random_append_matches_oracle(case):
    idx, fmt, dtype, B, C, paged, page, pos_hi, mag, eps, theta = case
    rng = np.random.default_rng(7000 + idx)
    dt = torch.float16 if dtype == "f16" else torch.bfloat16

    def draw(*shape, scale=mag):
        return torch.from_numpy(rng.standard_normal(shape) * scale).to(DEV).to(dt)

    qp, kp, vp = draw(B, 32, 128), draw(B, 8, 128), draw(B, 8, 128)
    wq, wk = (1 + draw(128, scale=0.1).float()).to(dt), (1 + draw(128, scale=0.1).float()).to(dt)
    pos = torch.from_numpy(rng.integers(0, pos_hi, B).astype(np.int32)).to(DEV)
    slots = torch.from_numpy(rng.integers(0, C, B).astype(np.int32)).to(DEV)
    w = inputs.custom(B, C, C, kv_dtype=fmt, q_dtype=dtype if fmt in ("e4m3", "i8") else None,
                      kv_std=2.0 if fmt == "e4m3" else 1.0, index=600 + idx)
    t = inputs.make(w, DEV)
    ks, vs = (t["k_scale"], t["v_scale"]) if fmt == "e4m3" else (1.0, 1.0)
    kv_bits0 = bits_of(t["kv"])
    sc_bits0 = bits_of(t["kv_scales"]) if fmt == "i8" else None
    if paged:
        pt = inputs.paginate(t, page, extra_pages=1, seed=idx)
        q_out = gq.append_kv_paged(qp, kp, vp, wq, wk, pos, slots, pt["kv_pages"], pt["block_table"], eps=eps,
                                   rope_theta=theta, k_scale=ks, v_scale=vs, kv_scales=pt.get("kv_scale_pages"))
        torch.cuda.synchronize()
        table, full = pt["block_table"].cpu().numpy(), np.full(B, C)
        kv_bits = oracle.gather_pages(bits_of(pt["kv_pages"]), table, full)
        sc_bits = oracle.gather_pages(bits_of(pt["kv_scale_pages"]), table, full) if fmt == "i8" else None
    else:
        q_out = gq.append_kv(qp, kp, vp, wq, wk, pos, slots, t["kv"], eps=eps, rope_theta=theta, k_scale=ks,
                             v_scale=vs, kv_scales=t["kv_scales"])
        torch.cuda.synchronize()
        kv_bits = bits_of(t["kv"])
        sc_bits = bits_of(t["kv_scales"]) if fmt == "i8" else None

    vals = lambda x: x.float().cpu().numpy().astype(np.float64)  # noqa: E731
    qo, ko, vo = oracle.append_kv(vals(qp), vals(kp), vals(vp), vals(wq), vals(wk), pos.cpu().numpy(), eps, theta)
    d_q = ulps_apart(bits_of(q_out), oracle.round_to(qo, FMT[dtype]))
    assert d_q.max() <= 1, f"append case {idx}: q_out {int(d_q.max())} ulps from the oracle"
    sl = slots.cpu().numpy()
    rows = np.arange(B)
    new = kv_bits[rows, :, :, sl]  # [B, 2, 8, 128]: the written rows
    if fmt in ("f16", "bf16"):
        d_k = ulps_apart(new[:, 0], oracle.round_to(ko, FMT[fmt]))
        assert d_k.max() <= 1, f"append case {idx}: k {int(d_k.max())} ulps from the oracle"
        assert np.array_equal(new[:, 1], bits_of(vp)), f"append case {idx}: v is not copied bit for bit"
    elif fmt == "e4m3":
        table = _e4m3_table()
        for plane, ref, scale in ((0, ko, ks), (1, vo, vs)):
            got = torch.from_numpy(new[:, plane].copy()).view(torch.float8_e4m3fn).double().numpy()
            i = np.searchsorted(table, ref / scale)
            lo, hi = table[np.clip(i - 1, 0, len(table) - 1)], table[np.clip(i, 0, len(table) - 1)]
            assert np.all((got == lo) | (got == hi)), f"append case {idx}: e4m3 plane {plane} off its bracket"
    else:
        new_sc = torch.from_numpy(sc_bits[rows, :, :, sl].view(np.int16)).view(torch.bfloat16).double().numpy()
        for plane, ref in ((0, ko), (1, vo)):
            amax = np.abs(ref).max(axis=2)  # [B, 8]
            np.testing.assert_allclose(new_sc[:, plane], amax / 127, rtol=2 ** -8)
            got = new[:, plane].view(np.int8).astype(np.float64) * new_sc[:, plane, :, None]
            assert np.all(np.abs(got - ref) <= 0.5 * new_sc[:, plane, :, None] * (1 + 1e-3) + 1e-30), \
                f"append case {idx}: int8 plane {plane} off by more than half a step"
    # nothing else in the cache (or its row scales) changed
    kv_bits[rows, :, :, sl] = kv_bits0[rows, :, :, sl]
    assert np.array_equal(kv_bits, kv_bits0), f"append case {idx}: bytes outside the written rows changed"
    if fmt == "i8":
        sc_bits[rows, :, :, sl] = sc_bits0[rows, :, :, sl]
        assert np.array_equal(sc_bits, sc_bits0), f"append case {idx}: row scales outside the written rows changed"
