"""PyTorch-facing calls with the same names as the C ABI.

Argument marshalling only: shapes are read from the tensors, output and
workspace tensors are allocated with torch, and the call goes through the C
library on the tensors' current CUDA stream. Every step of the attention runs
in the library's kernels.
"""

from __future__ import annotations

import ctypes
import math

import torch

from ._lib import FAError, check, lib


def _ptr(t: torch.Tensor | None):
    # the C signatures declare c_void_p: a plain int address (or None for NULL) is passed as is
    return None if t is None else t.data_ptr()


# the current stream's raw handle, without building a torch Stream object per call
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(t: torch.Tensor):
    if _raw_stream is not None:
        return _raw_stream(t.device.index)
    return torch.cuda.current_stream(t.device).cuda_stream


def _need(t: torch.Tensor, name: str, dtype, ndim: int):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {ndim}-D tensor")


def _on_current_device(t: torch.Tensor):
    """The library launches on the current CUDA device; tensors elsewhere would be read
    through another device's pointers."""
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"the tensors are on {t.device}, but the current CUDA device is "
                         f"cuda:{torch.cuda.current_device()} (use torch.cuda.device)")


def _check_qkv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor):
    """q [B][Hq][T][d], k and v [B][Hkv][S][d] on one device, the current one. The
    library takes every size from q and k, so v must match k exactly and q must share
    B and d."""
    if not (q.device == k.device == v.device):
        raise ValueError("q, k and v must be on one device")
    _on_current_device(q)
    if tuple(k.shape) != tuple(v.shape):
        raise ValueError(f"k and v must have one shape, got {tuple(k.shape)} and {tuple(v.shape)}")
    if q.shape[0] != k.shape[0] or q.shape[3] != k.shape[3]:
        raise ValueError(f"q {tuple(q.shape)} and k {tuple(k.shape)} must share batch and head dimension")


def _out(t, name: str, shape, dtype, like: torch.Tensor) -> torch.Tensor:
    """A caller's output tensor, checked (the library writes it through a bare pointer,
    so a smaller or strided tensor would be written past its end), or a new one."""
    if t is None:
        return torch.empty(shape, dtype=dtype, device=like.device)
    if not isinstance(t, torch.Tensor) or t.device != like.device:
        raise ValueError(f"{name} must be a tensor on {like.device}")
    if t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {dtype} tensor of shape {tuple(shape)}, "
                         f"got {t.dtype} {tuple(t.shape)}")
    return t


def fa_fwd(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None, want_lse: bool = True):
    """Prefill forward: q [B][Hq][T][d], k, v [B][Hkv][S][d] bf16 -> (o bf16, lse fp32 or None)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16, 4)
    _check_qkv(q, k, v)
    B, Hq, T, d = q.shape
    Hkv, S = k.shape[1], k.shape[2]
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = _out(out, "out", q.shape, torch.bfloat16, q)
    if want_lse or lse is not None:
        lse = _out(lse, "lse", (B, Hq, T), torch.float32, q)
    st = lib().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, T, S, d, scale, int(causal), _stream(q))
    check(st, "fa_fwd")
    return o, lse


def fa_fwd_f32(q, k, v, causal: bool = False, scale: float | None = None):
    """The same forward in fp32 on the CUDA cores: fp32 q, k, v -> (o fp32, lse fp32)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.float32, 4)
    _check_qkv(q, k, v)
    B, Hq, T, d = q.shape
    Hkv, S = k.shape[1], k.shape[2]
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, T), dtype=torch.float32, device=q.device)
    st = lib().fa_fwd_f32(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, T, S, d, scale, int(causal), _stream(q))
    check(st, "fa_fwd_f32")
    return o, lse


def _ws_bytes(workspace, nbytes: int, device) -> int:
    """Size in bytes of a caller's workspace tensor (any dtype), checked against what the call needs."""
    if workspace.device != torch.device(device) or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous tensor on the inputs' device")
    size = workspace.numel() * workspace.element_size()
    if size < nbytes:
        raise ValueError(f"workspace needs {nbytes} bytes, got {size}")
    return size


def fa_bwd_workspace_bytes(B: int, Hq: int, T: int) -> int:
    return int(lib().fa_bwd_workspace_bytes(B, Hq, T))


def fa_bwd(q, k, v, o, lse, d_o, causal: bool = False, scale: float | None = None, workspace=None,
           dq=None, dk=None, dv=None):
    """Backward: q, o, d_o [B][Hq][T][d], k, v [B][Hkv][S][d] bf16, lse [B][Hq][T] fp32
    (the forward's) -> (dq, dk, dv) bf16."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (d_o, "d_o")):
        _need(t, n, torch.bfloat16, 4)
    _need(lse, "lse", torch.float32, 3)
    _check_qkv(q, k, v)
    B, Hq, T, d = q.shape
    for t, n in ((o, "o"), (d_o, "d_o")):
        if t.device != q.device or tuple(t.shape) != tuple(q.shape):
            raise ValueError(f"{n} must have q's shape {tuple(q.shape)} on its device")
    if lse.device != q.device or tuple(lse.shape) != (B, Hq, T):
        raise ValueError(f"lse must be [B][Hq][T] = {(B, Hq, T)} on q's device")
    Hkv, S = k.shape[1], k.shape[2]
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    nbytes = fa_bwd_workspace_bytes(B, Hq, T)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    ws_bytes = _ws_bytes(workspace, nbytes, q.device)
    dq = _out(dq, "dq", q.shape, torch.bfloat16, q)
    dk = _out(dk, "dk", k.shape, torch.bfloat16, q)
    dv = _out(dv, "dv", v.shape, torch.bfloat16, q)
    st = lib().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(d_o), _ptr(dq), _ptr(dk), _ptr(dv), B, Hq,
                      Hkv, T, S, d, scale, int(causal), _ptr(workspace), ws_bytes, _stream(q))
    check(st, "fa_bwd")
    return dq, dk, dv


def fa_fwd_kv_outer_workspace_bytes(B: int, Hq: int, T: int, d: int) -> int:
    return int(lib().fa_fwd_kv_outer_workspace_bytes(B, Hq, T, d))


def fa_fwd_kv_outer(q, k, v, causal: bool = False, scale: float | None = None, row_bands: int = 1, workspace=None,
                    out=None, lse=None):
    """The forward in the FlashAttention-1 loop order (key tiles outer, running
    state through HBM): q [B][Hq][T][d], k, v [B][Hkv][S][d] bf16 -> (o, lse)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16, 4)
    _check_qkv(q, k, v)
    B, Hq, T, d = q.shape
    Hkv, S = k.shape[1], k.shape[2]
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    nbytes = fa_fwd_kv_outer_workspace_bytes(B, Hq, T, d)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    ws_bytes = _ws_bytes(workspace, nbytes, q.device)
    o = _out(out, "out", q.shape, torch.bfloat16, q)
    lse = _out(lse, "lse", (B, Hq, T), torch.float32, q)
    st = lib().fa_fwd_kv_outer(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, T, S, d, scale,
                               int(causal), int(row_bands), _ptr(workspace), ws_bytes, _stream(q))
    check(st, "fa_fwd_kv_outer")
    return o, lse


def fa_num_splits_heuristic(B: int, Hkv: int, S: int, num_sms: int) -> int:
    return int(lib().fa_num_splits_heuristic(B, Hkv, S, num_sms))


def fa_decode_workspace_bytes(B: int, Hq: int, T: int, d: int, num_splits: int) -> int:
    return int(lib().fa_decode_workspace_bytes(B, Hq, T, d, num_splits))


def fa_num_splits_prefill(B: int, Hq: int, Hkv: int, T: int, S: int, num_sms: int) -> int:
    return int(lib().fa_num_splits_prefill(B, Hq, Hkv, T, S, num_sms))


def fa_decode_num_splits(B: int, Hq: int, Hkv: int, T: int, S: int, paged: bool = False,
                         num_sms: int | None = None, device=None) -> int:
    """The split count the decode calls take for num_splits = 0 (chosen by the C library)."""
    if num_sms is None:
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        num_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    return int(lib().fa_decode_num_splits(B, Hq, Hkv, T, S, int(paged), int(num_sms)))


def _workspace(B, Hq, T, d, n, device, workspace):
    nbytes = fa_decode_workspace_bytes(B, Hq, T, d, n)
    if nbytes == 0:
        return None, 0
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
    return workspace, _ws_bytes(workspace, nbytes, device)


def fa_decode_splitkv(q, k, v, causal: bool = True, num_splits: int = 0, scale: float | None = None,
                      workspace=None, out=None, lse=None):
    """Split-KV decode: q [B][Hq][T][d], k, v [B][Hkv][S][d] bf16 -> (o, lse)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16, 4)
    _check_qkv(q, k, v)
    B, Hq, T, d = q.shape
    Hkv, S = k.shape[1], k.shape[2]
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    # the workspace is sized for the count the library takes; num_splits passes through as given
    n = int(num_splits) or fa_decode_num_splits(B, Hq, Hkv, T, S, False, device=q.device)
    ws, ws_bytes = _workspace(B, Hq, T, d, n, q.device, workspace)
    o = _out(out, "out", q.shape, torch.bfloat16, q)
    lse = _out(lse, "lse", (B, Hq, T), torch.float32, q)
    st = lib().fa_decode_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, T, S, d, scale,
                                 int(causal), int(num_splits), _ptr(ws), ws_bytes, _stream(q))
    check(st, "fa_decode_splitkv")
    return o, lse


def fa_decode_splitkv_static(q, k, v, causal: bool = True, num_splits: int = 0, scale: float | None = None,
                             out=None, lse=None):
    """Split-KV decode with the partials in the library's fixed 4 MiB device array
    (no workspace, no allocation inside the call); see include/fa_gb300.h."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16, 4)
    _check_qkv(q, k, v)
    B, Hq, T, d = q.shape
    Hkv, S = k.shape[1], k.shape[2]
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = _out(out, "out", q.shape, torch.bfloat16, q)
    lse = _out(lse, "lse", (B, Hq, T), torch.float32, q)
    st = lib().fa_decode_splitkv_static(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, T, S, d, scale,
                                        int(causal), int(num_splits), _stream(q))
    check(st, "fa_decode_splitkv_static")
    return o, lse


def fa_lse_merge(o_part, lse_part):
    """Merge o_part [n][rows][d] fp32 and lse_part [n][rows] fp32 -> (o [rows][d] bf16, lse [rows] fp32)."""
    _need(o_part, "o_part", torch.float32, 3)
    _need(lse_part, "lse_part", torch.float32, 2)
    n, rows, d = o_part.shape
    if tuple(lse_part.shape) != (n, rows) or lse_part.device != o_part.device:
        raise ValueError("lse_part must be [n][rows] on o_part's device")
    _on_current_device(o_part)
    o = torch.empty((rows, d), dtype=torch.bfloat16, device=o_part.device)
    lse = torch.empty((rows,), dtype=torch.float32, device=o_part.device)
    st = lib().fa_lse_merge(_ptr(o_part), _ptr(lse_part), _ptr(o), _ptr(lse), n, rows, d, _stream(o_part))
    check(st, "fa_lse_merge")
    return o, lse


def fa_decode_paged(q, k_pages, v_pages, block_table, seqlens, causal: bool = True, num_splits: int = 0,
                    scale: float | None = None, workspace=None, out=None, lse=None):
    """Paged decode: pools [P][16][Hkv][d] bf16, block_table [B][max_pages] int32, seqlens [B] int32."""
    _need(q, "q", torch.bfloat16, 4)
    _need(k_pages, "k_pages", torch.bfloat16, 4)
    _need(v_pages, "v_pages", torch.bfloat16, 4)
    _need(block_table, "block_table", torch.int32, 2)
    _need(seqlens, "seqlens", torch.int32, 1)
    B, Hq, T, d = q.shape
    P, page_size, Hkv, _ = k_pages.shape
    max_pages = block_table.shape[1]
    if not (q.device == k_pages.device == v_pages.device == block_table.device == seqlens.device):
        raise ValueError("q, the pools, block_table and seqlens must be on one device")
    _on_current_device(q)
    if tuple(k_pages.shape) != tuple(v_pages.shape) or k_pages.shape[3] != d:
        raise ValueError(f"k_pages and v_pages must both be [P][page_size][Hkv][{d}]")
    if block_table.shape[0] != B or tuple(seqlens.shape) != (B,):
        raise ValueError(f"block_table must be [{B}][max_pages] and seqlens [{B}]")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    n = int(num_splits) or fa_decode_num_splits(B, Hq, Hkv, T, max_pages * page_size, True, device=q.device)
    ws, ws_bytes = _workspace(B, Hq, T, d, n, q.device, workspace)
    o = _out(out, "out", q.shape, torch.bfloat16, q)
    lse = _out(lse, "lse", (B, Hq, T), torch.float32, q)
    st = lib().fa_decode_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table), _ptr(seqlens), _ptr(o),
                               _ptr(lse), B, Hq, Hkv, T, max_pages, page_size, P, d, scale, int(causal),
                               int(num_splits), _ptr(ws), ws_bytes, _stream(q))
    check(st, "fa_decode_paged")
    return o, lse


def fa_get_last_device_error(device=None) -> tuple[int, int]:
    """Synchronise the current stream and read/clear the device error word -> (status, raw word)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    detail = ctypes.c_int(0)
    st = lib().fa_get_last_device_error(ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream), ctypes.byref(detail))
    return int(st), int(detail.value)


def fa_set_wait_timeout_ns(ns: int) -> None:
    lib().fa_set_wait_timeout_ns(int(ns))


def fa_get_wait_timeouts() -> tuple[int, int]:
    """(bound of the waits between roles, bound of the waits before a CTA exits), in ns."""
    w, u = ctypes.c_ulonglong(0), ctypes.c_ulonglong(0)
    lib().fa_get_wait_timeouts(ctypes.byref(w), ctypes.byref(u))
    return int(w.value), int(u.value)


def fa_selftest_wait_timeout(timeout_ns: int, device=None) -> None:
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    st = lib().fa_selftest_wait_timeout(int(timeout_ns), ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream))
    check(st, "fa_selftest_wait_timeout")


__all__ = [
    "FAError",
    "fa_fwd",
    "fa_fwd_f32",
    "fa_bwd",
    "fa_bwd_workspace_bytes",
    "fa_num_splits_heuristic",
    "fa_num_splits_prefill",
    "fa_decode_num_splits",
    "fa_decode_workspace_bytes",
    "fa_decode_splitkv",
    "fa_decode_splitkv_static",
    "fa_lse_merge",
    "fa_decode_paged",
    "fa_get_last_device_error",
    "fa_set_wait_timeout_ns",
    "fa_get_wait_timeouts",
    "fa_selftest_wait_timeout",
]
