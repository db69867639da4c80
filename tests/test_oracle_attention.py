"""Pins for the oracle's attention arithmetic.

Each test checks the FP64 oracle against something other than itself: exact
rational answers of hand-built cases (tests/golden/worked_examples.json),
closed forms (length 1 gives V[0]; q_scale = 0 or equal keys give the mean of
V; a very large q_scale gives the value row of the largest score), invariants
of softmax attention (slot permutation, a common shift of every key, the
convex hull of the value rows, power-of-two scaling of V, k_scale and q_scale
acting only through their product), the grouped head map, torch's float64
scaled_dot_product_attention on the dequantised inputs, and a brute-force
restatement in 40-digit decimal arithmetic on tiny caches.
"""
import decimal
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from gqa_decode_attention_sm_gb300 import inputs
from helpers import D, HKV, HQ, bits_of, f16_bits, bf16_bits, sdpa_f64, values_of_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")
FMT = {"f16": oracle.F16, "bf16": oracle.BF16, "e4m3": oracle.E4M3, "i8": oracle.I8}


def _to_bits(vals, fmt):
    return f16_bits(vals) if fmt == "f16" else bf16_bits(vals)


def _explicit(lib, q_vals, k_vals, v_vals, lens, fmt="f16", **kw):
    """Run the oracle on explicit values (exactly representable in ``fmt``)."""
    qb = _to_bits(q_vals, fmt)
    kv = np.stack([k_vals, v_vals], axis=1)  # [B,2,8,C,128]
    kvb = _to_bits(kv, fmt)
    assert np.array_equal(values_of_bits(kvb, fmt), kv), "test values must be exact"
    return oracle.gqa_decode(qb, FMT[fmt], kvb, FMT[fmt], np.asarray(lens, np.int32), lib=lib,
                             **kw)


def _random(w, seed=None):
    t = inputs.make(w, "cpu", seed=seed)
    return t, bits_of(t["q"]), bits_of(t["kv"]), t["lens"].numpy()


def _run(lib, t, qb, kvb, lens, **kw):
    w = t["workload"]
    args = dict(q_scale=t["q_scale"], k_scale=t["k_scale"], v_scale=t["v_scale"])
    if t.get("kv_scales") is not None:
        args["kv_scales"] = bits_of(t["kv_scales"])
    args.update(kw)
    return oracle.gqa_decode(qb, FMT[w.q_dtype], kvb, FMT[w.kv_dtype], lens, lib=lib, **args)


# ------------------------------------------------- brute force, 40 digits


def _brute_force_decimal(q_vals, k_vals, v_vals, lens, q_scale, k_scale, v_scale):
    """Softmax attention written out in decimal arithmetic at 40 digits from
    the decoded values (exact binary fractions, so Decimal(x) is exact)."""
    ctx = decimal.Context(prec=40)
    Dd = decimal.Decimal
    B = q_vals.shape[0]
    scale = ctx.divide(ctx.multiply(Dd(q_scale), Dd(k_scale)), ctx.sqrt(Dd(D)))
    out = np.zeros((B * HQ, D))
    for b in range(B):
        L = int(lens[b])
        for h in range(HQ):
            g = h // (HQ // HKV)
            s = []
            for t in range(L):
                acc = Dd(0)
                for d in range(D):
                    acc = ctx.add(acc, ctx.multiply(Dd(float(q_vals[b, h, d])), Dd(float(k_vals[b, g, t, d]))))
                s.append(ctx.multiply(scale, acc))
            m = max(s)
            w = [ctx.exp(ctx.subtract(x, m)) for x in s]
            den = sum(w, Dd(0))
            for d in range(D):
                num = sum((ctx.multiply(w[t], Dd(float(v_vals[b, g, t, d]))) for t in range(L)), Dd(0))
                out[b * HQ + h, d] = float(ctx.multiply(Dd(v_scale), ctx.divide(num, den)))
    return out


@pytest.mark.parametrize("fmt", ["f16", "bf16", "e4m3"])
def test_matches_40_digit_brute_force_on_tiny_caches(orc, fmt):
    rng = np.random.default_rng({"f16": 1, "bf16": 2, "e4m3": 3}[fmt])
    B, C = 2, 8
    q_fmt = "bf16" if fmt == "e4m3" else fmt
    qv = rng.standard_normal((B, HQ, D)) * 1.5
    qb = f16_bits(qv) if q_fmt == "f16" else bf16_bits(qv)
    kv = rng.standard_normal((B, 2, HKV, C, D)) * 2.0
    if fmt == "e4m3":
        kvb = torch.from_numpy(kv.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        k_scale, v_scale = 0.75, 1.25  # distinct, both applied
    else:
        kvb = _to_bits(kv, fmt)
        k_scale = v_scale = 1.0
    lens = np.array([int(rng.integers(1, C + 1)), C], dtype=np.int32)
    q_scale = 0.8
    got, _ = oracle.gqa_decode(qb, FMT[q_fmt], kvb, FMT[fmt], lens, q_scale=q_scale, k_scale=k_scale,
                               v_scale=v_scale, lib=orc)
    q_vals = values_of_bits(qb, q_fmt)
    kv_vals = values_of_bits(kvb, fmt)
    want = _brute_force_decimal(q_vals, kv_vals[:, 0], kv_vals[:, 1], lens, q_scale, k_scale, v_scale)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-14)


# ------------------------------------------------------------------ golden


def test_golden_worked_examples(orc):
    spec = json.load(open(GOLDEN))
    q_scale = math.log(2.0) * math.sqrt(128.0) / 8.0
    for case in spec["cases"]:
        L = len(case["k_dim0"])
        C = L + 3
        q = np.zeros((1, HQ, D)); q[0, :, 0] = 1.0
        k = np.zeros((1, HKV, C, D)); v = np.zeros((1, HKV, C, D))
        k[0, :, :L, 0] = case["k_dim0"]
        vv = np.asarray(case["v"], dtype=np.float64)
        v[0, :, :L, :vv.shape[1]] = vv
        k[0, :, L:, :] = np.nan  # slots past the length hold NaN; they must not be read
        v[0, :, L:, :] = np.nan
        qb = f16_bits(q)
        kvb = f16_bits(np.stack([k, v], axis=1))
        out, _ = oracle.gqa_decode(qb, oracle.F16, kvb, oracle.F16, np.array([L], np.int32),
                                   q_scale=q_scale, lib=orc)
        want = [float(Fraction(x)) for x in case["expected"]]
        for h in range(HQ):
            np.testing.assert_allclose(out[h, :len(want)], want, rtol=1e-13, atol=1e-15,
                                       err_msg=case["name"])
            assert np.all(out[h, len(want):] == 0.0)


# ------------------------------------------------------------- closed forms


@pytest.mark.parametrize("kv_dtype", ["f16", "bf16", "e4m3"])
def test_length_one_returns_first_value_row(orc, kv_dtype):
    w = inputs.custom(3, 16, 1, kv_dtype=kv_dtype, nan_tail=True)
    t, qb, kvb, lens = _random(w)
    out, bits = _run(orc, t, qb, kvb, lens)
    vals = values_of_bits(kvb, kv_dtype)
    for r in range(3 * HQ):
        b, h = divmod(r, HQ)
        v0 = vals[b, 1, h // 4, 0] * t["v_scale"]
        assert np.array_equal(out[r], v0)
        if kv_dtype != "e4m3":  # V[0] is representable in the output type
            assert np.array_equal(bits[r], kvb[b, 1, h // 4, 0])


@pytest.mark.parametrize("kv_dtype", ["f16", "bf16", "e4m3"])
def test_zero_q_scale_gives_mean_of_values(orc, kv_dtype):
    w = inputs.custom(2, 96, 40, 96, kv_dtype=kv_dtype)
    t, qb, kvb, lens = _random(w)
    out, _ = _run(orc, t, qb, kvb, lens, q_scale=0.0)
    vals = values_of_bits(kvb, kv_dtype)
    for r in range(2 * HQ):
        b, h = divmod(r, HQ)
        L = lens[b]
        mean = [math.fsum(vals[b, 1, h // 4, :L, d]) / L * t["v_scale"] for d in range(D)]
        np.testing.assert_allclose(out[r], mean, rtol=1e-12, atol=1e-14)


def test_equal_keys_give_mean_of_values(orc):
    rng = np.random.default_rng(11)
    B, C, L = 2, 48, 37
    q = rng.integers(-3, 4, (B, HQ, D)).astype(np.float64)
    k = np.repeat(rng.integers(-3, 4, (B, HKV, 1, D)), C, axis=2).astype(np.float64)
    v = rng.integers(-8, 9, (B, HKV, C, D)).astype(np.float64)
    out, _ = _explicit(orc, q, k, v, [L, L])
    for r in range(B * HQ):
        b, h = divmod(r, HQ)
        want = [math.fsum(v[b, h // 4, :L, d]) / L for d in range(D)]
        np.testing.assert_allclose(out[r], want, rtol=1e-13, atol=1e-14)


def test_large_q_scale_selects_largest_score(orc):
    # k_t = t * e0 and q = e0: the score grows with t, so the limit is V[L-1]
    B, C, L = 1, 32, 20
    q = np.zeros((B, HQ, D)); q[..., 0] = 1.0
    k = np.zeros((B, HKV, C, D)); k[0, :, :, 0] = np.arange(C)
    v = np.random.default_rng(2).integers(-50, 50, (B, HKV, C, D)).astype(np.float64)
    out, _ = _explicit(orc, q, k, v, [L], q_scale=2000.0)  # adjacent weights differ by e^-177
    for h in range(HQ):
        np.testing.assert_allclose(out[h], v[0, h // 4, L - 1], rtol=1e-14, atol=1e-14)


def test_grouped_head_map(orc):
    # every V row of KV head g equals g+1, so query head h must return h//4 + 1
    rng = np.random.default_rng(5)
    B, C = 2, 24
    q = rng.integers(-4, 5, (B, HQ, D)).astype(np.float64)
    k = rng.integers(-4, 5, (B, HKV, C, D)).astype(np.float64)
    v = np.broadcast_to((np.arange(HKV) + 1.0)[None, :, None, None], (B, HKV, C, D)).copy()
    out, _ = _explicit(orc, q, k, v, [C, 9])
    for r in range(B * HQ):
        np.testing.assert_allclose(out[r], (r % HQ) // 4 + 1.0, rtol=1e-14)


# --------------------------------------------------------------- invariants


def test_permuting_slots_leaves_output_unchanged(orc):
    w = inputs.custom(2, 80, 60, 80)
    t, qb, kvb, lens = _random(w)
    ref, _ = _run(orc, t, qb, kvb, lens)
    rng = np.random.default_rng(9)
    kvp = kvb.copy()
    for b in range(2):
        L = lens[b]
        perm = rng.permutation(L)
        kvp[b, :, :, :L] = np.take(kvb[b], perm, axis=2)
    got, _ = _run(orc, t, qb, kvp, lens)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)


def test_common_key_shift_leaves_output_unchanged(orc):
    rng = np.random.default_rng(12)
    B, C = 1, 40
    q = (rng.integers(-8, 9, (B, HQ, D)) / 8.0)
    k = rng.integers(-6, 7, (B, HKV, C, D)).astype(np.float64)
    v = rng.integers(-6, 7, (B, HKV, C, D)).astype(np.float64)
    shift = rng.integers(-5, 6, (B, HKV, 1, D)).astype(np.float64)
    a, _ = _explicit(orc, q, k, v, [C])
    b, _ = _explicit(orc, q, k + shift, v, [C])
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-14)


def test_output_inside_convex_hull_of_values(orc):
    w = inputs.custom(4, 64, 1, 64)
    t, qb, kvb, lens = _random(w, seed=77)
    out, _ = _run(orc, t, qb, kvb, lens, q_scale=3.0)
    vals = values_of_bits(kvb, "f16")
    for r in range(4 * HQ):
        b, h = divmod(r, HQ)
        vv = vals[b, 1, h // 4, :lens[b]]
        assert np.all(out[r] >= vv.min(axis=0) - 1e-12) and np.all(out[r] <= vv.max(axis=0) + 1e-12)


def test_slots_past_length_are_never_read(orc):
    w = inputs.custom(4, 128, 1, 127)
    t, qb, kvb, lens = _random(w, seed=3)
    kv_nan = t["kv"].clone(); inputs.fill_tail(kv_nan, lens, "f16", float("nan"))
    kv_big = t["kv"].clone(); inputs.fill_tail(kv_big, lens, "f16", 60000.0)
    a, abits = _run(orc, t, qb, bits_of(kv_nan), lens)
    b, bbits = _run(orc, t, qb, bits_of(kv_big), lens)
    assert np.array_equal(a, b) and np.array_equal(abits, bbits) and np.isfinite(a).all()


def test_v_scale_is_linear_and_k_scale_folds_into_q_scale(orc):
    w = inputs.custom(2, 64, 30, 64, kv_dtype="e4m3", kv_std=2.0)
    t, qb, kvb, lens = _random(w)
    base, _ = _run(orc, t, qb, kvb, lens, q_scale=0.75, k_scale=0.5, v_scale=1.0)
    scaled, _ = _run(orc, t, qb, kvb, lens, q_scale=0.75, k_scale=0.5, v_scale=4.0)
    assert np.array_equal(scaled, 4.0 * base)  # power-of-two scaling is exact
    folded, _ = _run(orc, t, qb, kvb, lens, q_scale=0.375, k_scale=1.0, v_scale=1.0)
    np.testing.assert_allclose(base, folded, rtol=1e-12, atol=1e-14)
    other, _ = _run(orc, t, qb, kvb, lens, q_scale=0.75, k_scale=1.0, v_scale=1.0)
    assert not np.allclose(base, other, rtol=1e-6)  # k_scale really changes the scores


def test_rejects_lengths_outside_capacity(orc):
    w = inputs.custom(2, 16, 4)
    t, qb, kvb, _ = _random(w)
    for bad in ([0, 4], [4, 17], [-1, 4]):
        with pytest.raises(ValueError):
            _run(orc, t, qb, kvb, np.array(bad, np.int32))


# -------------------------------------------------- library special case


def _check_sdpa(orc, t, qb, kvb, lens, rows=None, **kw):
    w = t["workload"]
    out, bits = _run(orc, t, qb, kvb, lens, rows=rows, **kw)
    qv = values_of_bits(qb, w.q_dtype)
    kvv = values_of_bits(kvb, w.kv_dtype)
    if w.kv_dtype == "i8":  # dequantise: code x the bf16 scale of its row
        kvv = kvv * t["kv_scales"].to(torch.float64).numpy()[..., None]
    args = dict(q_scale=t["q_scale"], k_scale=t["k_scale"], v_scale=t["v_scale"])
    args.update(kw)
    ref = sdpa_f64(qv, kvv[:, 0], kvv[:, 1], lens, rows=rows, **args)
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)
    # the single rounding step agrees with the reference value rounded by numpy/torch
    ref_t = torch.from_numpy(ref)
    if w.q_dtype == "f16":
        assert np.mean(bits == ref.astype(np.float16).view(np.uint16)) > 0.999
    else:
        rb = ref_t.to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.mean(bits == rb) > 0.999


@pytest.mark.parametrize("index", [1, 2])
def test_matches_torch_sdpa_on_small_workloads(orc, index):
    t, qb, kvb, lens = _random(inputs.WORKLOADS[index])
    _check_sdpa(orc, t, qb, kvb, lens)


def test_matches_torch_sdpa_on_ragged_nan_tail_sample(orc):
    # the ragged workload's recipe (NaN tails, U[1,C] lengths) at a smaller capacity
    w = inputs.with_(inputs.WORKLOADS[3], capacity=1024, len_hi=1024, batch=8)
    t, qb, kvb, lens = _random(w)
    _check_sdpa(orc, t, qb, kvb, lens, rows=list(range(0, 8 * HQ, 5)))


def test_matches_torch_sdpa_fp8_with_distinct_scales(orc):
    w = inputs.custom(3, 200, 50, 200, kv_dtype="e4m3", kv_std=2.0)
    t, qb, kvb, lens = _random(w)
    _check_sdpa(orc, t, qb, kvb, lens, q_scale=1.0, k_scale=t["k_scale"] * 0.5,
                v_scale=t["v_scale"] * 3.0)


# ------------------------------------------------------------ INT8 cache


def test_int8_length_one_returns_scaled_first_row(orc):
    w = inputs.custom(3, 16, 1, kv_dtype="i8", nan_tail=True)
    t, qb, kvb, lens = _random(w)
    out, _ = _run(orc, t, qb, kvb, lens)
    codes = kvb.view(np.int8).astype(np.float64)
    scales = t["kv_scales"].to(torch.float64).numpy()
    for r in range(3 * HQ):
        b, h = divmod(r, HQ)
        assert np.array_equal(out[r], codes[b, 1, h // 4, 0] * scales[b, 1, h // 4, 0])


def test_int8_matches_torch_sdpa_on_dequantised_rows(orc):
    w = inputs.custom(3, 200, 50, 200, kv_dtype="i8", nan_tail=True)
    t, qb, kvb, lens = _random(w)
    _check_sdpa(orc, t, qb, kvb, lens)


def test_int8_scales_act_per_row(orc):
    # codes c with row scale s, or codes 2c with row scale s/2: the same values,
    # so the same output (exactly); a different scale on one V row changes it
    rng = np.random.default_rng(21)
    B, C, L = 1, 24, 20
    t = inputs.make(inputs.custom(B, C, L, kv_dtype="i8"), "cpu")
    codes = rng.integers(-63, 64, (B, 2, 8, C, 128)).astype(np.int8)
    scales = np.exp2(rng.integers(-8, -2, (B, 2, 8, C))).astype(np.float32)
    qb = bits_of(t["q"])
    lens = np.array([L], np.int32)

    def run(c, s):
        return oracle.gqa_decode(qb, oracle.BF16, c.view(np.uint8), oracle.I8, lens, lib=orc,
                                 kv_scales=bf16_bits(s))[0]

    a = run(codes, scales)
    b = run((codes.astype(np.int16) * 2).astype(np.int8), scales / 2)
    assert np.array_equal(a, b)
    s2 = scales.copy()
    s2[0, 1, :, 3] *= 2
    assert not np.allclose(run(codes, s2), a, rtol=1e-9)


# ------------------------------------------------------------- paged cache


@pytest.mark.parametrize("page_size", [16, 64])
def test_paged_gather_reproduces_the_contiguous_cache(orc, page_size):
    w = inputs.custom(3, 256, 1, 256, nan_tail=True)
    t, qb, kvb, lens = _random(w, seed=5)
    pt = inputs.paginate(t, page_size, extra_pages=4, seed=9)
    g = oracle.gather_pages(bits_of(pt["kv_pages"]), pt["block_table"].numpy(), lens)
    for b in range(3):  # every slot below the length comes back in place
        assert np.array_equal(g[b, :, :, :lens[b]], kvb[b, :, :, :lens[b]])
    a, _ = _run(orc, t, qb, kvb, lens)
    c, _ = _run(orc, t, qb, g, lens)
    assert np.array_equal(a, c)


@pytest.mark.parametrize("page_size", [16, 64])
def test_paged_gather_of_an_int8_cache_and_its_scale_pool(orc, page_size):
    w = inputs.custom(3, 256, 1, 256, kv_dtype="i8", nan_tail=True)
    t, qb, kvb, lens = _random(w, seed=6)
    pt = inputs.paginate(t, page_size, extra_pages=4, seed=10)
    g = oracle.gather_pages(bits_of(pt["kv_pages"]), pt["block_table"].numpy(), lens)
    gs = oracle.gather_pages(bits_of(pt["kv_scale_pages"]), pt["block_table"].numpy(), lens)
    sc = bits_of(t["kv_scales"])
    for b in range(3):
        assert np.array_equal(g[b, :, :, :lens[b]], kvb[b, :, :, :lens[b]])
        assert np.array_equal(gs[b, :, :, :lens[b]], sc[b, :, :, :lens[b]])
    a, _ = _run(orc, t, qb, kvb, lens)
    c, _ = _run(orc, t, qb, g, lens, kv_scales=gs)
    assert np.array_equal(a, c)


# ----------------------------------------------------------- verify window


def _window_sdpa(t):
    """torch float64 SDPA with an explicit causal mask over the window."""
    w = t["workload"]
    T = w.q_len
    qv = values_of_bits(bits_of(t["q"]), w.q_dtype)            # [B,T,32,128]
    kvv = values_of_bits(bits_of(t["kv"]), w.kv_dtype)         # [B,2,8,C,128]
    lens = t["lens"].numpy()
    out = np.zeros((w.batch, T, HQ, D))
    for b in range(w.batch):
        L = int(lens[b])
        q = torch.from_numpy(np.ascontiguousarray(qv[b].transpose(1, 0, 2)))[None]  # [1,32,T,128]
        k = torch.from_numpy(np.ascontiguousarray(kvv[b, 0, :, :L])).repeat_interleave(4, 0)[None]
        v = torch.from_numpy(np.ascontiguousarray(kvv[b, 1, :, :L])).repeat_interleave(4, 0)[None]
        mask = torch.arange(L)[None, :] <= (L - T + torch.arange(T))[:, None]          # [T,L]
        o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask,
                                                             scale=t["q_scale"] / math.sqrt(D))
        out[b] = o[0].numpy().transpose(1, 0, 2)
    return out.reshape(-1, D)


@pytest.mark.parametrize("T", [2, 3, 4])
def test_window_matches_torch_sdpa_with_causal_mask(orc, T):
    w = inputs.custom(2, 128, 4, 128, kv_dtype="bf16", q_len=T, nan_tail=True)
    t, qb, kvb, lens = _random(w, seed=30 + T)
    out, _ = _run(orc, t, qb, kvb, lens)
    np.testing.assert_allclose(out, _window_sdpa(t), rtol=1e-10, atol=1e-12)


def test_window_2(orc):
    test_window_matches_torch_sdpa_with_causal_mask(orc, 2)


def test_window_rows_are_single_token_problems(orc):
    # query j of a T-token window equals a one-token decode over the first L-T+1+j slots
    T = 3
    w = inputs.custom(2, 64, 10, 64, q_len=T)
    t, qb, kvb, lens = _random(w, seed=4)
    out, _ = _run(orc, t, qb, kvb, lens)
    for b in range(2):
        for j in range(T):
            one, _ = oracle.gqa_decode(qb[b:b + 1, j], oracle.F16, kvb[b:b + 1], oracle.F16,
                                       np.array([lens[b] - T + 1 + j], np.int32), lib=orc)
            r0 = (b * T + j) * HQ
            assert np.array_equal(out[r0:r0 + HQ], one)


def test_window_rejects_lengths_below_q_len(orc):
    w = inputs.custom(2, 16, 4, q_len=4)
    t, qb, kvb, _ = _random(w)
    with pytest.raises(ValueError):
        _run(orc, t, qb, kvb, np.array([3, 4], np.int32))
