"""Seeded synthetic inputs for GQA decode attention.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic.  Both the CUDA path's tests/bench and the CPU oracle take
their inputs from here.

Workloads (shapes, distributions and structure of the five decode cases):
  1  fp16  batch 1,  capacity 64,     lengths 64
  2  fp16  batch 1,  capacity 1024,   lengths 1024
  3  fp16  batch 32, capacity 8192,   lengths U[1,8192], slots >= length hold NaN
  4  bf16  batch 8,  capacity 131072, lengths 131072
  5  bf16 q, e4m3 KV, batch 64, capacity 32768, lengths U[16384,32768];
     K,V ~ N(0,1)*2 quantised with one per-tensor scale amax/448
q ~ N(0,1) everywhere; K,V ~ N(0,1) for workloads 1-4; q_scale = 1.

An INT8 cache (kv_dtype "i8") stores int8 codes with one bf16 scale per
(plane, KV head, position) row: scale = amax(|row|)/127 rounded to bf16,
code = round(x / scale) clipped to [-127, 127].

Recipe: a torch.Generator on the target device; lengths drawn first from
``seed``; q from ``seed + 1``; the KV slice of batch row b from
``seed * 7919 + 1000 + b`` so rows can be generated (and regenerated) one at a
time without holding an fp32 copy of the whole cache.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch

HQ, HKV, D = 32, 8, 128
E4M3_MAX = 448.0


@dataclass(frozen=True)
class Workload:
    index: int
    name: str
    kv_dtype: str          # "f16" | "bf16" | "e4m3" | "i8"
    q_dtype: str           # "f16" | "bf16"
    batch: int
    capacity: int
    len_lo: int            # lengths ~ U[len_lo, len_hi] (inclusive); equal => constant
    len_hi: int
    nan_tail: bool = False  # fill K/V slots >= length with NaN
    kv_std: float = 1.0
    q_scale: float = 1.0
    q_len: int = 1          # query tokens per request (a verify window when > 1)

    @property
    def seed(self) -> int:
        return 1000 + self.index


WORKLOADS = {
    1: Workload(1, "fp16 B1 C64 L64", "f16", "f16", 1, 64, 64, 64),
    2: Workload(2, "fp16 B1 C1024 L1024", "f16", "f16", 1, 1024, 1024, 1024),
    3: Workload(3, "fp16 B32 C8192 ragged U[1,8192] NaN tail", "f16", "f16", 32, 8192, 1, 8192,
                nan_tail=True),
    4: Workload(4, "bf16 B8 C131072 L131072", "bf16", "bf16", 8, 131072, 131072, 131072),
    5: Workload(5, "e4m3 KV bf16 q B64 C32768 U[16384,32768]", "e4m3", "bf16", 64, 32768,
                16384, 32768, kv_std=2.0),
}


def custom(batch: int, capacity: int, len_lo: int, len_hi: int | None = None,
           kv_dtype: str = "f16", q_dtype: str | None = None, nan_tail: bool = False,
           kv_std: float = 1.0, q_scale: float = 1.0, index: int = 0, q_len: int = 1) -> Workload:
    """A workload of any size with the same recipe (edge cases, small tests)."""
    if q_dtype is None:
        q_dtype = "bf16" if kv_dtype in ("e4m3", "i8") else kv_dtype
    return Workload(index, f"custom B{batch} C{capacity}", kv_dtype, q_dtype, batch, capacity,
                    len_lo, len_lo if len_hi is None else len_hi, nan_tail, kv_std, q_scale, q_len)


_TORCH = {"f16": torch.float16, "bf16": torch.bfloat16}


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def kv_storage_dtype(w: Workload) -> torch.dtype:
    if w.kv_dtype == "e4m3":
        return torch.uint8
    if w.kv_dtype == "i8":
        return torch.int8
    return _TORCH[w.kv_dtype]


def _kv_row_fp32(w: Workload, b: int, device, seed: int) -> torch.Tensor:
    g = _gen(device, seed * 7919 + 1000 + b)
    x = torch.randn((2, HKV, w.capacity, D), generator=g, device=device, dtype=torch.float32)
    if w.kv_std != 1.0:
        x.mul_(w.kv_std)
    return x


def make(w: Workload, device="cpu", seed: int | None = None, lens=None) -> dict:
    """Build one batch of inputs on ``device``.

    Returns a dict with q [B,32,128] ([B,q_len,32,128] for a verify window),
    kv [B,2,8,C,128] (uint8 bytes for e4m3,
    int8 codes for i8), kv_scales (bf16 [B,2,8,C] for i8, else None), lens
    int32 [B], q_scale, k_scale, v_scale (python floats; the e4m3 scale is the
    fp32 value actually stored), and the workload.
    ``lens`` overrides the drawn lengths (a list or tensor of B ints).
    """
    seed = w.seed if seed is None else int(seed)
    device = torch.device(device)
    B, C = w.batch, w.capacity
    if lens is None:
        if w.len_lo == w.len_hi:
            lens_t = torch.full((B,), w.len_lo, dtype=torch.int32)
        else:
            lens_t = torch.randint(w.len_lo, w.len_hi + 1, (B,), generator=_gen("cpu", seed),
                                   dtype=torch.int64).to(torch.int32)
    else:
        lens_t = torch.as_tensor(lens, dtype=torch.int32).reshape(B).clone()
    q_shape = (B, HQ, D) if w.q_len == 1 else (B, w.q_len, HQ, D)
    q = torch.randn(q_shape, generator=_gen(device, seed + 1), device=device,
                    dtype=torch.float32).to(_TORCH[w.q_dtype])

    kv = torch.empty((B, 2, HKV, C, D), device=device, dtype=kv_storage_dtype(w))
    k_scale = v_scale = 1.0
    kv_scales = None
    if w.kv_dtype == "i8":
        kv_scales = torch.empty((B, 2, HKV, C), device=device, dtype=torch.bfloat16)
        for b in range(B):
            x = _kv_row_fp32(w, b, device, seed)
            sc = (x.abs().amax(dim=-1) / 127.0).to(torch.bfloat16)   # one scale per row
            sc = torch.where(sc == 0, torch.ones_like(sc), sc)
            codes = torch.round(x / sc.float().unsqueeze(-1)).clamp_(-127, 127)
            kv[b].copy_(codes.to(torch.int8))
            kv_scales[b].copy_(sc)
    elif w.kv_dtype == "e4m3":
        # one amax over every K and V value of the allocated cache
        amax = torch.zeros((), device=device, dtype=torch.float32)
        for b in range(B):
            amax = torch.maximum(amax, _kv_row_fp32(w, b, device, seed).abs().amax())
        scale = (amax / E4M3_MAX).to(torch.float32)
        k_scale = v_scale = float(scale.item())
        for b in range(B):
            x = _kv_row_fp32(w, b, device, seed).div_(scale)
            kv[b].copy_(x.to(torch.float8_e4m3fn).view(torch.uint8))
    else:
        for b in range(B):
            kv[b].copy_(_kv_row_fp32(w, b, device, seed).to(_TORCH[w.kv_dtype]))
    if w.nan_tail:
        fill_tail(kv, lens_t, w.kv_dtype)
        if kv_scales is not None:  # codes have no NaN: poison the unused rows' scales instead
            for b, L in enumerate(lens_t.tolist()):
                kv_scales[b, :, :, L:] = float("nan")
    return dict(q=q, kv=kv, lens=lens_t.to(device), q_scale=w.q_scale, k_scale=k_scale,
                v_scale=v_scale, kv_scales=kv_scales, workload=w)


def make_row(w: Workload, b: int, device="cpu", seed: int | None = None) -> dict:
    """Batch row ``b`` of ``make(w)``, drawn from the same generators without
    building the other rows: q [1,32,128], kv [1,2,8,C,128], lens [1].

    Only the 16-bit formats (f16, bf16): the e4m3 recipe needs one amax over
    the whole cache.  Lets a CPU test use one row of a multi-GB workload."""
    if w.kv_dtype not in _TORCH:
        raise ValueError("make_row draws 16-bit caches only")
    seed = w.seed if seed is None else int(seed)
    device = torch.device(device)
    B = w.batch
    if w.len_lo == w.len_hi:
        lens_t = torch.full((B,), w.len_lo, dtype=torch.int32)
    else:
        lens_t = torch.randint(w.len_lo, w.len_hi + 1, (B,), generator=_gen("cpu", seed),
                               dtype=torch.int64).to(torch.int32)
    q_shape = (B, HQ, D) if w.q_len == 1 else (B, w.q_len, HQ, D)
    q = torch.randn(q_shape, generator=_gen(device, seed + 1), device=device,
                    dtype=torch.float32).to(_TORCH[w.q_dtype])
    kv = _kv_row_fp32(w, b, device, seed).to(_TORCH[w.kv_dtype]).unsqueeze(0)
    lens_b = lens_t[b:b + 1].clone()
    if w.nan_tail:
        fill_tail(kv, lens_b, w.kv_dtype)
    return dict(q=q[b:b + 1].clone(), kv=kv, lens=lens_b.to(device), q_scale=w.q_scale, k_scale=1.0,
                v_scale=1.0, kv_scales=None, workload=w)


def fill_tail(kv: torch.Tensor, lens, kv_dtype: str, value: float = float("nan")) -> None:
    """Overwrite every K and V slot t >= lens[b] with ``value`` (NaN by default).

    For e4m3 bytes NaN is the pattern 0x7F (S.1111.111); other values are cast.
    """
    lens_l = [int(x) for x in torch.as_tensor(lens).cpu().tolist()]
    for b, L in enumerate(lens_l):
        if L >= kv.shape[3]:
            continue
        if kv_dtype == "i8":  # codes cannot hold NaN: use the extreme code
            kv[b, :, :, L:, :].fill_(-128 if value != value else int(max(-127, min(127, value))))
        elif kv_dtype == "e4m3":
            if value != value:  # NaN
                kv[b, :, :, L:, :].fill_(0x7F)
            else:
                t = torch.tensor(value, dtype=torch.float32).to(torch.float8_e4m3fn)
                kv[b, :, :, L:, :].fill_(int(t.view(torch.uint8).item()))
        else:
            kv[b, :, :, L:, :].fill_(value)


def bits(t: torch.Tensor):
    """Raw bit patterns of a tensor as numpy (uint16 for 2-byte types, uint8 bytes)."""
    t = t.detach().contiguous()
    if t.dtype in (torch.float16, torch.bfloat16):
        return t.view(torch.int16).cpu().numpy().view("uint16")
    if t.dtype == torch.uint8:
        return t.cpu().numpy()
    if t.dtype == torch.int8:
        return t.cpu().numpy().view("uint8")
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).cpu().numpy()
    raise TypeError(f"no bit view for {t.dtype}")


def with_(w: Workload, **kw) -> Workload:
    return replace(w, **kw)


def paginate(t: dict, page_size: int, extra_pages: int = 3, seed: int = 0) -> dict:
    """Scatter a contiguous cache into a shuffled page pool (a paged cache).

    Returns a copy of ``t`` with kv_pages [num_pages, 2, 8, page_size, 128]
    (same dtype), block_table int32 [B, C/page_size] and num_pages; an int8
    cache also gets kv_scale_pages bf16 [num_pages, 2, 8, page_size].  Page
    ids are a seeded permutation; ``extra_pages`` spare pages, and the
    block-table entries of pages past each length, point at pages filled with
    NaN (0x7F for e4m3 bytes, -128 codes with NaN scales for int8), which a
    correct kernel never reads.
    """
    kv = t["kv"]
    B, _, H, C, Dd = kv.shape
    assert C % page_size == 0, "capacity must be a whole number of pages"
    per = C // page_size
    lens = [int(x) for x in t["lens"].cpu().tolist()]
    used = [(b, j) for b in range(B) for j in range(per) if j * page_size < lens[b]]
    num_pages = len(used) + extra_pages
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) + 77)
    ids = torch.randperm(num_pages, generator=g)
    pages = torch.empty((num_pages, 2, H, page_size, Dd), dtype=kv.dtype, device=kv.device)
    if kv.dtype == torch.uint8:
        pages.fill_(0x7F)
    elif kv.dtype == torch.int8:
        pages.fill_(-128)
    else:
        pages.fill_(float("nan"))
    scales = t.get("kv_scales")
    spages = None
    if scales is not None:
        spages = torch.full((num_pages, 2, H, page_size), float("nan"), dtype=scales.dtype, device=kv.device)
    spare = [int(x) for x in ids[len(used):]] or [int(ids[0])]
    table = torch.full((B, per), spare[0], dtype=torch.int32)
    for n, (b, j) in enumerate(used):
        pid = int(ids[n])
        table[b, j] = pid
        pages[pid].copy_(kv[b, :, :, j * page_size:(j + 1) * page_size, :])
        if spages is not None:
            spages[pid].copy_(scales[b, :, :, j * page_size:(j + 1) * page_size])
    out = dict(t)
    out.update(kv_pages=pages, block_table=table.to(kv.device), num_pages=num_pages, page_size=page_size,
               kv_scale_pages=spages)
    return out
