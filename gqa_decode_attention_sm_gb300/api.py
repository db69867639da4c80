"""Thin PyTorch-facing binding over the C ABI (argument marshalling only).

Mirrors the three calls of the "FlashInfer sm110_gqa_decode" article
(sections "Convenience API" and "Prepared continuous decoding"):
``gqa_decode`` (convenience), ``prepare`` + ``launch`` (prepared: validation
and workspace allocation happen once, the launch allocates nothing and can be
captured in a CUDA graph), plus ``gqa_decode_fp8kv`` for an e4m3 KV cache
(the "FP8 KV cache port on Jetson AGX Thor" blog: uint8 cache bytes are
reinterpreted as float8_e4m3fn; k_scale on the scores, v_scale on the output).
Every step of the computation runs in the library's CUDA kernels; PyTorch only
provides device memory and the current stream.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import torch

from . import _lib
from ._lib import GqaError

HQ, HKV, D = 32, 8, 128
F16, BF16 = 0, 1
KV_F16, KV_BF16, KV_E4M3, KV_I8 = 0, 1, 2, 3
MAX_SPLITS = 256
FLAG_LENGTH_CLAMPED = 0x1
FLAG_WAIT_TIMEOUT = 0x2
FLAG_PAGE_CLAMPED = 0x4
FLAG_SLOT_CLAMPED = 0x8
FLAG_BOUNDS = 0x10  # range-checked build only: an access fell outside its buffer

_QDT = {torch.float16: F16, torch.bfloat16: BF16}
_KVF = {torch.float16: KV_F16, torch.bfloat16: KV_BF16, torch.uint8: KV_E4M3,
        torch.float8_e4m3fn: KV_E4M3, torch.int8: KV_I8}

__all__ = ["GqaError", "append_kv_paged", "gqa_decode", "gqa_decode_fp8kv", "gqa_decode_int8kv", "gqa_decode_paged",
           "gqa_decode_verify", "append_kv",
           "prepare", "launch",
           "Prepared",
           "workspace_size", "plan", "get_status", "split_stage", "combine_stage", "split_geometry",
           "launch_count"]


def _ptr(t: torch.Tensor) -> int:
    return t.data_ptr()


def _stream(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _require(t, name, shape, dtypes, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype not in dtypes:
        raise ValueError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def _geometry(q, kv, lens):
    _require(q, "q", None, (torch.float16, torch.bfloat16))
    if q.dim() != 3 or q.shape[1:] != (HQ, D):
        raise ValueError(f"q must be [batch, {HQ}, {D}], got {tuple(q.shape)}")
    B = q.shape[0]
    if kv.dim() != 5 or kv.shape[0] != B or kv.shape[1:3] != (2, HKV) or kv.shape[4] != D:
        raise ValueError(f"kv must be [{B}, 2, {HKV}, capacity, {D}], got {tuple(kv.shape)}")
    C = kv.shape[3]
    _require(kv, "kv", None, tuple(_KVF), q.device)
    _require(lens, "sequence_lengths", (B,), (torch.int32,), q.device)
    return B, C


def workspace_size(batch: int, capacity: int, num_splits: int) -> int:
    n = _lib.load().gqa_decode_workspace_size(batch, capacity, num_splits)
    if n == 0:
        raise ValueError("invalid batch/capacity/num_splits")
    return int(n)


def plan(batch: int, capacity: int, kv_format: int, device=None) -> int:
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    out = ctypes.c_int(0)
    _lib.check(_lib.load().gqa_decode_plan(batch, capacity, kv_format, dev.index or 0,
                                           ctypes.byref(out)))
    return out.value


def split_geometry(capacity: int, num_splits: int, kv_format: int):
    """(tokens per split, number of splits holding slots) for this geometry."""
    chunk, eff = ctypes.c_int(0), ctypes.c_int(0)
    _lib.check(_lib.load().gqa_decode_split_geometry(capacity, num_splits, kv_format,
                                                     ctypes.byref(chunk), ctypes.byref(eff)))
    return chunk.value, eff.value


def launch_count(batch: int, capacity: int, kv_format: int, q_len: int, num_splits: int, sm_count: int) -> int:
    """Kernels one decode call of these sizes enqueues: 1 (one split, or the
    splits merged on chip in a thread-block cluster) or 2 (split + combine)."""
    out = ctypes.c_int(0)
    _lib.check(_lib.load().gqa_decode_launch_count_for(batch, capacity, kv_format, q_len, num_splits, sm_count,
                                                       ctypes.byref(out)))
    return out.value


def gqa_decode(q, kv, sequence_lengths, q_scale: float = 1.0, out=None):
    """Convenience call: plans, takes a stream-ordered workspace, launches."""
    B, C = _geometry(q, kv, sequence_lengths)
    if kv.dtype != q.dtype:
        raise ValueError("kv must have the dtype of q (use gqa_decode_fp8kv for e4m3)")
    if out is None:
        out = torch.empty_like(q)
    _require(out, "out", q.shape, (q.dtype,), q.device)
    with torch.cuda.device(q.device):
        _lib.check(_lib.load().gqa_decode(_ptr(q), _ptr(kv), _ptr(sequence_lengths), _ptr(out), B, C,
                                          _QDT[q.dtype], float(q_scale), _stream(q.device)))
    return out


@dataclass
class Prepared:
    """Everything a launch needs, validated once.  Keep it (and its tensors)
    alive until every launch or graph replay that uses it has finished.  One
    Prepared per concurrently running stream/graph: its workspace is mutable."""
    q: torch.Tensor
    kv: torch.Tensor
    out: torch.Tensor
    lens: torch.Tensor
    workspace: torch.Tensor
    batch: int
    capacity: int
    q_dtype: int
    kv_format: int
    q_scale: float
    k_scale: float
    v_scale: float
    num_splits: int
    kv_scales: torch.Tensor | None = None  # int8 cache: bf16 [B,2,8,C]

    @property
    def workspace_bytes(self) -> int:
        return self.workspace.numel()

    @property
    def splits_effective(self) -> int:
        return split_geometry(self.capacity, self.num_splits, self.kv_format)[1]


def _storage_overlaps(a: torch.Tensor, b: torch.Tensor) -> bool:
    sa, sb = a.untyped_storage(), b.untyped_storage()
    x0, y0 = sa.data_ptr(), sb.data_ptr()
    return x0 < y0 + sb.nbytes() and y0 < x0 + sa.nbytes()


def prepare(tensors: dict, q_scale: float = 1.0, num_splits=None, k_scale=None, v_scale=None,
            workspace: torch.Tensor | None = None) -> Prepared:
    """Validate once and allocate the split workspace once (outside any capture).

    ``tensors`` holds "Q", "KV", "O", "sequence_lengths", and "KV_SCALES" for an
    int8 cache.  An e4m3 cache (uint8 or float8_e4m3fn storage) needs k_scale
    and v_scale.  A ``workspace`` given by the caller (uint8, at least
    workspace_size bytes) should have its 256-byte header (status flags) zeroed
    before first use (``workspace_init``).
    """
    q, kv, out, lens = tensors["Q"], tensors["KV"], tensors["O"], tensors["sequence_lengths"]
    B, C = _geometry(q, kv, lens)
    kv_scales = tensors.get("KV_SCALES")
    if kv.dtype == torch.int8:
        _require(kv_scales, "KV_SCALES", (B, 2, HKV, C), (torch.bfloat16,), q.device)
    _require(out, "O", q.shape, (q.dtype,), q.device)
    for name, t in (("Q", q), ("KV", kv), ("sequence_lengths", lens), ("KV_SCALES", kv_scales)):
        if t is not None and _storage_overlaps(out, t):
            raise ValueError(f"O must not share storage with {name}")
    kvf = _KVF[kv.dtype]
    if kvf not in (KV_E4M3, KV_I8) and kv.dtype != q.dtype:
        raise ValueError("fp16/bf16 KV must have the dtype of Q")
    if kvf == KV_E4M3:
        if k_scale is None or v_scale is None:
            raise ValueError("an e4m3 KV cache needs k_scale and v_scale")
    else:
        k_scale = 1.0 if k_scale is None else k_scale
        v_scale = 1.0 if v_scale is None else v_scale
    if not (float(q_scale) > 0.0 and float(q_scale) < float("inf")):
        raise ValueError("q_scale must be finite and > 0")
    S = plan(B, C, kvf, q.device) if not num_splits else int(num_splits)
    nbytes = workspace_size(B, C, S)
    if workspace is None:
        workspace = torch.zeros(nbytes, dtype=torch.uint8, device=q.device)
    else:
        _require(workspace, "workspace", None, (torch.uint8,), q.device)
        if workspace.numel() < nbytes:
            raise ValueError(f"workspace has {workspace.numel()} bytes, needs {nbytes}")
    return Prepared(q, kv, out, lens, workspace, B, C, _QDT[q.dtype], kvf, float(q_scale),
                    float(k_scale), float(v_scale), S, kv_scales if kvf == KV_I8 else None)


def launch(p: Prepared) -> torch.Tensor:
    """Run both stages on the current stream: no allocation, no host read."""
    lib = _lib.load()
    with torch.cuda.device(p.q.device):
        st = _stream(p.q.device)
        if p.kv_format == KV_I8:
            _lib.check(lib.gqa_decode_int8kv(_ptr(p.q), _ptr(p.kv), _ptr(p.kv_scales), _ptr(p.lens),
                                             _ptr(p.out), p.batch, p.capacity, p.q_dtype, p.q_scale,
                                             p.num_splits, _ptr(p.workspace), p.workspace_bytes, st))
        elif p.kv_format == KV_E4M3 and p.q_dtype == BF16:
            _lib.check(lib.gqa_decode_fp8kv(_ptr(p.q), _ptr(p.kv), _ptr(p.lens), _ptr(p.out), p.batch,
                                            p.capacity, p.q_scale, p.k_scale, p.v_scale, p.num_splits,
                                            _ptr(p.workspace), p.workspace_bytes, st))
        elif p.kv_format == KV_E4M3:
            split_stage(p)
            combine_stage(p)
        else:
            _lib.check(lib.gqa_decode_prepared(_ptr(p.q), _ptr(p.kv), _ptr(p.lens), _ptr(p.out), p.batch,
                                               p.capacity, p.q_dtype, p.q_scale, p.num_splits,
                                               _ptr(p.workspace), p.workspace_bytes, st))
    return p.out


def split_stage(p: Prepared) -> None:
    """Stage 1 alone (streams K/V, writes partials or, with one split, out).
    Not for an int8 cache (its scales go through gqa_decode_int8kv)."""
    with torch.cuda.device(p.q.device):
        _lib.check(_lib.load().gqa_decode_split_stage(
            _ptr(p.q), p.q_dtype, _ptr(p.kv), p.kv_format, _ptr(p.lens), _ptr(p.out), p.batch,
            p.capacity, p.q_scale, p.k_scale, p.v_scale, p.num_splits, _ptr(p.workspace),
            p.workspace_bytes, _stream(p.q.device)))


def combine_stage(p: Prepared) -> None:
    """Stage 2 alone (log-sum-exp merge of the partials; nothing with one split)."""
    with torch.cuda.device(p.q.device):
        _lib.check(_lib.load().gqa_decode_combine_stage(
            _ptr(p.lens), _ptr(p.out), p.q_dtype, p.kv_format, p.batch, p.capacity, p.v_scale,
            p.num_splits, _ptr(p.workspace), p.workspace_bytes, _stream(p.q.device)))


def gqa_decode_fp8kv(q, kv, sequence_lengths, k_scale: float, v_scale: float, q_scale: float = 1.0,
                     out=None, num_splits=None, workspace=None):
    """e4m3 KV cache (uint8 or float8_e4m3fn storage), bf16 q and out."""
    B, C = _geometry(q, kv, sequence_lengths)
    if q.dtype != torch.bfloat16 or _KVF[kv.dtype] != KV_E4M3:
        raise ValueError("gqa_decode_fp8kv takes bf16 q and an e4m3 (uint8) KV cache")
    if out is None:
        out = torch.empty_like(q)
    _require(out, "out", q.shape, (torch.bfloat16,), q.device)
    S = plan(B, C, KV_E4M3, q.device) if not num_splits else int(num_splits)
    nbytes = workspace_size(B, C, S)
    if workspace is None:
        workspace = torch.zeros(nbytes, dtype=torch.uint8, device=q.device)
    with torch.cuda.device(q.device):
        _lib.check(_lib.load().gqa_decode_fp8kv(
            _ptr(q), _ptr(kv), _ptr(sequence_lengths), _ptr(out), B, C, float(q_scale), float(k_scale),
            float(v_scale), S, _ptr(workspace), workspace.numel(), _stream(q.device)))
    return out


def gqa_decode_int8kv(q, kv, kv_scales, sequence_lengths, q_scale: float = 1.0, out=None,
                      num_splits=None, workspace=None):
    """int8 cache with one bf16 scale per (plane, KV head, slot) row; fp16/bf16 q and out."""
    B, C = _geometry(q, kv, sequence_lengths)
    if kv.dtype != torch.int8:
        raise ValueError("gqa_decode_int8kv takes an int8 KV cache")
    _require(kv_scales, "kv_scales", (B, 2, HKV, C), (torch.bfloat16,), q.device)
    if out is None:
        out = torch.empty_like(q)
    _require(out, "out", q.shape, (q.dtype,), q.device)
    S = plan(B, C, KV_I8, q.device) if not num_splits else int(num_splits)
    nbytes = workspace_size(B, C, S)
    if workspace is None:
        workspace = torch.zeros(nbytes, dtype=torch.uint8, device=q.device)
    with torch.cuda.device(q.device):
        _lib.check(_lib.load().gqa_decode_int8kv(
            _ptr(q), _ptr(kv), _ptr(kv_scales), _ptr(sequence_lengths), _ptr(out), B, C, _QDT[q.dtype],
            float(q_scale), S, _ptr(workspace), workspace.numel(), _stream(q.device)))
    return out


def gqa_decode_paged(q, kv_pages, block_table, sequence_lengths, q_scale: float = 1.0,
                     k_scale: float = 1.0, v_scale: float = 1.0, out=None, num_splits=None,
                     workspace=None, kv_scales=None):
    """Paged cache: kv_pages [num_pages, 2, 8, page_size, 128] (fp16/bf16, e4m3 as
    uint8/float8_e4m3fn, or int8 with kv_scales bf16 [num_pages, 2, 8, page_size]),
    block_table int32 [batch, max_pages]; q [batch, 32, 128], or [batch, T, 32, 128]
    for a verify window of T = 1..4 tokens; returns out (q's shape)."""
    _require(q, "q", None, (torch.float16, torch.bfloat16))
    B = q.shape[0]
    if q.dim() == 3 and q.shape[1:] == (HQ, D):
        T = 1
    elif q.dim() == 4 and q.shape[2:] == (HQ, D) and 1 <= q.shape[1] <= 4:
        T = q.shape[1]
    else:
        raise ValueError(f"q must be [batch, {HQ}, {D}] or [batch, T (1..4), {HQ}, {D}]")
    if kv_pages.dim() != 5 or kv_pages.shape[1:3] != (2, HKV) or kv_pages.shape[4] != D:
        raise ValueError("kv_pages must be [num_pages, 2, 8, page_size, 128]")
    _require(kv_pages, "kv_pages", None, tuple(_KVF), q.device)
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table must be [batch, max_pages]")
    _require(block_table, "block_table", None, (torch.int32,), q.device)
    _require(sequence_lengths, "sequence_lengths", (B,), (torch.int32,), q.device)
    kvf = _KVF[kv_pages.dtype]
    num_pages, page_size, max_pages = kv_pages.shape[0], kv_pages.shape[3], block_table.shape[1]
    if kvf == KV_I8:
        _require(kv_scales, "kv_scales", (num_pages, 2, HKV, page_size), (torch.bfloat16,), q.device)
    C = max_pages * page_size
    if out is None:
        out = torch.empty_like(q)
    _require(out, "out", q.shape, (q.dtype,), q.device)
    S = plan(B, C, kvf, q.device) if not num_splits else int(num_splits)
    nbytes = workspace_size(B * T, C, S)
    if workspace is None:
        workspace = torch.zeros(nbytes, dtype=torch.uint8, device=q.device)
    with torch.cuda.device(q.device):
        _lib.check(_lib.load().gqa_decode_paged(
            _ptr(q), _QDT[q.dtype], _ptr(kv_pages), kvf, _ptr(kv_scales) if kvf == KV_I8 else None,
            _ptr(block_table), max_pages, num_pages, page_size, _ptr(sequence_lengths), _ptr(out), B, T,
            float(q_scale), float(k_scale), float(v_scale), S, _ptr(workspace), workspace.numel(),
            _stream(q.device)))
    return out


def gqa_decode_verify(q, kv, sequence_lengths, q_scale: float = 1.0, k_scale: float = 1.0,
                      v_scale: float = 1.0, kv_scales=None, out=None, num_splits=None, workspace=None):
    """Verify window: q [batch, T, 32, 128] (T = 1..4 draft tokens, the last T slots
    of each cache row); query j attends slots [0, len - T + j].  Any KV format
    (int8 needs kv_scales).  Returns out [batch, T, 32, 128]."""
    _require(q, "q", None, (torch.float16, torch.bfloat16))
    if q.dim() != 4 or q.shape[2:] != (HQ, D):
        raise ValueError(f"q must be [batch, T, {HQ}, {D}], got {tuple(q.shape)}")
    B, T = q.shape[0], q.shape[1]
    if kv.dim() != 5 or kv.shape[0] != B or kv.shape[1:3] != (2, HKV) or kv.shape[4] != D:
        raise ValueError(f"kv must be [{B}, 2, {HKV}, capacity, {D}]")
    C = kv.shape[3]
    _require(kv, "kv", None, tuple(_KVF), q.device)
    _require(sequence_lengths, "sequence_lengths", (B,), (torch.int32,), q.device)
    kvf = _KVF[kv.dtype]
    if kvf == KV_I8:
        _require(kv_scales, "kv_scales", (B, 2, HKV, C), (torch.bfloat16,), q.device)
    if out is None:
        out = torch.empty_like(q)
    _require(out, "out", q.shape, (q.dtype,), q.device)
    S = plan(B, C, kvf, q.device) if not num_splits else int(num_splits)
    nbytes = workspace_size(B * T, C, S)
    if workspace is None:
        workspace = torch.zeros(nbytes, dtype=torch.uint8, device=q.device)
    with torch.cuda.device(q.device):
        _lib.check(_lib.load().gqa_decode_verify(
            _ptr(q), _QDT[q.dtype], _ptr(kv), kvf, _ptr(kv_scales) if kvf == KV_I8 else None,
            _ptr(sequence_lengths), _ptr(out), B, C, T, float(q_scale), float(k_scale), float(v_scale), S,
            _ptr(workspace), workspace.numel(), _stream(q.device)))
    return out


def append_kv(q_proj, k_proj, v_proj, q_norm_w, k_norm_w, positions, slots, kv, q_out=None,
              eps: float = 1e-6, rope_theta: float = 1e6, k_scale: float = 1.0, v_scale: float = 1.0,
              kv_scales=None, workspace=None):
    """RMS norm + RoPE of the new token's q and k heads; k and v written into
    ``kv`` at ``slots``; returns q_out [batch, 32, 128] ready for decode."""
    _require(q_proj, "q_proj", None, (torch.float16, torch.bfloat16))
    B = q_proj.shape[0]
    dt = q_proj.dtype
    _require(q_proj, "q_proj", (B, HQ, D), (dt,))
    _require(k_proj, "k_proj", (B, HKV, D), (dt,), q_proj.device)
    _require(v_proj, "v_proj", (B, HKV, D), (dt,), q_proj.device)
    _require(q_norm_w, "q_norm_w", (D,), (dt,), q_proj.device)
    _require(k_norm_w, "k_norm_w", (D,), (dt,), q_proj.device)
    _require(positions, "positions", (B,), (torch.int32,), q_proj.device)
    _require(slots, "slots", (B,), (torch.int32,), q_proj.device)
    if kv.dim() != 5 or kv.shape[0] != B or kv.shape[1:3] != (2, HKV) or kv.shape[4] != D:
        raise ValueError(f"kv must be [{B}, 2, {HKV}, capacity, {D}]")
    _require(kv, "kv", None, tuple(_KVF), q_proj.device)
    kvf = _KVF[kv.dtype]
    if q_out is None:
        q_out = torch.empty_like(q_proj)
    _require(q_out, "q_out", q_proj.shape, (dt,), q_proj.device)
    with torch.cuda.device(q_proj.device):
        _lib.check(_lib.load().gqa_append_kv(
            _ptr(q_proj), _ptr(k_proj), _ptr(v_proj), _ptr(q_norm_w), _ptr(k_norm_w), _QDT[dt],
            _ptr(positions), _ptr(slots), B, _ptr(q_out), _ptr(kv), kvf,
            _ptr(kv_scales) if kv_scales is not None else None, kv.shape[3], float(eps), float(rope_theta),
            float(k_scale), float(v_scale), _ptr(workspace) if workspace is not None else None,
            workspace.numel() if workspace is not None else 0, _stream(q_proj.device)))
    return q_out


def append_kv_paged(q_proj, k_proj, v_proj, q_norm_w, k_norm_w, positions, slots, kv_pages, block_table,
                    q_out=None, eps: float = 1e-6, rope_theta: float = 1e6, k_scale: float = 1.0,
                    v_scale: float = 1.0, kv_scales=None, workspace=None):
    """append_kv on a paged cache: kv_pages [num_pages, 2, 8, page_size, 128] (and,
    for int8, kv_scales [num_pages, 2, 8, page_size] bf16), block_table int32
    [batch, max_pages]; slot s of row b lands in row s % page_size of page
    block_table[b, s // page_size]."""
    _require(q_proj, "q_proj", None, (torch.float16, torch.bfloat16))
    B = q_proj.shape[0]
    dt = q_proj.dtype
    _require(q_proj, "q_proj", (B, HQ, D), (dt,))
    _require(k_proj, "k_proj", (B, HKV, D), (dt,), q_proj.device)
    _require(v_proj, "v_proj", (B, HKV, D), (dt,), q_proj.device)
    _require(q_norm_w, "q_norm_w", (D,), (dt,), q_proj.device)
    _require(k_norm_w, "k_norm_w", (D,), (dt,), q_proj.device)
    _require(positions, "positions", (B,), (torch.int32,), q_proj.device)
    _require(slots, "slots", (B,), (torch.int32,), q_proj.device)
    if kv_pages.dim() != 5 or kv_pages.shape[1:3] != (2, HKV) or kv_pages.shape[4] != D:
        raise ValueError("kv_pages must be [num_pages, 2, 8, page_size, 128]")
    _require(kv_pages, "kv_pages", None, tuple(_KVF), q_proj.device)
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table must be [batch, max_pages]")
    _require(block_table, "block_table", None, (torch.int32,), q_proj.device)
    kvf = _KVF[kv_pages.dtype]
    num_pages, page_size = kv_pages.shape[0], kv_pages.shape[3]
    if kvf == KV_I8:
        _require(kv_scales, "kv_scales", (num_pages, 2, HKV, page_size), (torch.bfloat16,), q_proj.device)
    if q_out is None:
        q_out = torch.empty_like(q_proj)
    _require(q_out, "q_out", q_proj.shape, (dt,), q_proj.device)
    with torch.cuda.device(q_proj.device):
        _lib.check(_lib.load().gqa_append_kv_paged(
            _ptr(q_proj), _ptr(k_proj), _ptr(v_proj), _ptr(q_norm_w), _ptr(k_norm_w), _QDT[dt],
            _ptr(positions), _ptr(slots), B, _ptr(q_out), _ptr(kv_pages), kvf,
            _ptr(kv_scales) if kv_scales is not None else None, _ptr(block_table), block_table.shape[1],
            num_pages, page_size, float(eps), float(rope_theta), float(k_scale), float(v_scale),
            _ptr(workspace) if workspace is not None else None,
            workspace.numel() if workspace is not None else 0, _stream(q_proj.device)))
    return q_out


def workspace_init(workspace: torch.Tensor) -> None:
    """Zero a workspace's header (status flags) on the current stream."""
    with torch.cuda.device(workspace.device):
        _lib.check(_lib.load().gqa_decode_workspace_init(_ptr(workspace), workspace.numel(),
                                                         _stream(workspace.device)))


def get_status(p_or_workspace) -> int:
    """Debug only (synchronises): read and clear the workspace status flags."""
    ws = p_or_workspace.workspace if isinstance(p_or_workspace, Prepared) else p_or_workspace
    flags = ctypes.c_uint32(0)
    with torch.cuda.device(ws.device):
        _lib.check(_lib.load().gqa_decode_get_status(_ptr(ws), ws.numel(), _stream(ws.device),
                                                     ctypes.byref(flags)))
    return flags.value
