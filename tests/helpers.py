"""Shared test helpers: building small inputs from explicit values, bit views,
and the library special case (torch float64 scaled_dot_product_attention).

Nothing here computes attention except ``sdpa_f64``, which is torch's own
routine called on the dequantised inputs (a library special case, used as a pin
for the oracle), and ``tolerance_ok``, the parity bar.
"""
import math

import numpy as np
import torch

HQ, HKV, D = 32, 8, 128

# GPU vs oracle bar: |gpu - ref| <= 3e-3, or relative 1e-2 where |ref| > 0.3
ABS_TOL = 3e-3
REL_TOL = 1e-2
REL_FLOOR = 0.3


def f16_bits(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)


def bf16_bits(x) -> np.ndarray:
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_of(t: torch.Tensor) -> np.ndarray:
    t = t.detach().contiguous().cpu()
    if t.dtype in (torch.float16, torch.bfloat16):
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.uint8:
        return t.numpy()
    if t.dtype == torch.int8:
        return t.numpy().view(np.uint8)
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    raise TypeError(t.dtype)


def values_of_bits(b: np.ndarray, fmt: str) -> np.ndarray:
    """Library decode (torch) of raw bits to float64."""
    if fmt == "f16":
        return b.view(np.float16).astype(np.float64)
    if fmt == "bf16":
        return torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    if fmt == "e4m3":
        return torch.from_numpy(b).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    if fmt == "i8":  # the codes only (the row scales are separate)
        return b.view(np.int8).astype(np.float64)
    raise ValueError(fmt)


def sdpa_f64(q_vals, k_vals, v_vals, lens, q_scale=1.0, k_scale=1.0, v_scale=1.0, rows=None):
    """torch float64 SDPA with K/V repeated per query head (repeat_interleave(4)).

    q_vals [B,32,128], k_vals/v_vals [B,8,C,128] float64 arrays.  Returns [n_rows,128].
    """
    B = q_vals.shape[0]
    rows = list(range(B * HQ)) if rows is None else list(rows)
    out = np.zeros((len(rows), D))
    by_b = {}
    for i, r in enumerate(rows):
        by_b.setdefault(r // HQ, []).append((i, r % HQ))
    for b, items in by_b.items():
        L = int(lens[b])
        q = torch.from_numpy(np.ascontiguousarray(q_vals[b])).reshape(1, HQ, 1, D)
        k = torch.from_numpy(np.ascontiguousarray(k_vals[b, :, :L])) * k_scale
        v = torch.from_numpy(np.ascontiguousarray(v_vals[b, :, :L])) * v_scale
        k = k.repeat_interleave(HQ // HKV, dim=0).unsqueeze(0)
        v = v.repeat_interleave(HQ // HKV, dim=0).unsqueeze(0)
        o = torch.nn.functional.scaled_dot_product_attention(
            q, k, v, scale=q_scale / math.sqrt(D))[0, :, 0, :].numpy()
        for i, h in items:
            out[i] = o[h]
    return out


def tolerance_ok(got: np.ndarray, ref: np.ndarray):
    """Element-wise parity bar; returns (ok, worst abs error, worst excess)."""
    err = np.abs(got - ref)
    allowed = np.where(np.abs(ref) > REL_FLOOR, np.maximum(ABS_TOL, REL_TOL * np.abs(ref)), ABS_TOL)
    excess = err - allowed
    return bool(np.all(excess <= 0) and np.all(np.isfinite(got))), float(err.max()), float(excess.max())


# Second gate for long contexts.  There the outputs are averages of many V
# rows and shrink like 1/sqrt(length) (about 4.6e-3 RMS at 131072 tokens), so
# the absolute 3e-3 bar is most of the signal and would pass an output that
# lost a whole split of the sequence (such a loss moves it by roughly
# RMS / sqrt(splits)).  The kernels' own errors are about 1-2 % of the RMS,
# set by the final fp16/bf16 rounding and the 16-bit softmax weights.
RMS_GATE = 0.05


def rms_gate_ok(got: np.ndarray, ref: np.ndarray, frac: float = RMS_GATE):
    """max |got - ref| <= frac * RMS(ref); returns (ok, max error / RMS(ref))."""
    rms = float(np.sqrt(np.mean(np.square(ref))))
    err = float(np.max(np.abs(got - ref)))
    ratio = err / rms if rms > 0 else (0.0 if err == 0 else float("inf"))
    return bool(ratio <= frac and np.all(np.isfinite(got))), ratio


def ulps_apart(got_bits, ref_bits) -> np.ndarray:
    """Distance in units in the last place between 16-bit float patterns of
    the same format (ordered by value; +0 and -0 coincide)."""
    def ordered(b):
        b = np.asarray(b, dtype=np.int64)
        mag = b & 0x7FFF
        return np.where(b & 0x8000, -mag, mag)
    return np.abs(ordered(got_bits) - ordered(ref_bits))
