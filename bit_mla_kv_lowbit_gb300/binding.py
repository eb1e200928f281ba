"""ctypes binding of ``libmla_lowbit.so`` (the C ABI in include/mla_lowbit.h).

Argument marshalling only: each function checks tensor devices, dtypes,
shapes and contiguity, then passes raw pointers and the current CUDA stream
to the library.  Every step of the computation runs in the library's CUDA
kernels; there is no fallback, and loading fails loudly when the library is
missing.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

from . import build as _build

_LIB: Optional[ctypes.CDLL] = None

EXPORTS = (
    "mla_lowbit_page_bytes",
    "mla_lowbit_bytes_per_token",
    "mla_lowbit_write",
    "mla_lowbit_decode_plan",
    "mla_lowbit_decode",
    "mla_lowbit_decode_noalloc",
    "mla_lowbit_write_decode",
    "mla_lowbit_decode_multi",
    "mla_lowbit_set_fault_injection",
    "mla_lowbit_read_error",
    "mla_lowbit_strerror",
    "mla_lowbit_version",
)

DEV_BAD_SEQ, DEV_BAD_POS, DEV_BAD_PAGE, DEV_BAD_LEN, DEV_PLAN, DEV_PIPELINE = 1, 2, 4, 8, 16, 32


class Layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("content_bits", "rope_bits", "group", "sink", "local", "page_tokens",
                 "latent", "rope", "rotate")]


def layout(content_bits: int = 4, rope_bits: int = 4, rotate: bool = False) -> Layout:
    return Layout(content_bits, rope_bits, 64, 4, 128, 64, 512, 64, int(bool(rotate)))


class LibraryError(RuntimeError):
    pass


def lib_path() -> str:
    return _build.LIB


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load the library (building it first if it is missing or stale)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = path or lib_path()
    if not os.path.exists(path):
        _build.build_library()
    if not os.path.exists(path):
        raise LibraryError(f"libmla_lowbit.so not found at {path}")
    lib = ctypes.CDLL(path)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    lp = ctypes.POINTER(Layout)
    lib.mla_lowbit_page_bytes.argtypes = [lp]
    lib.mla_lowbit_page_bytes.restype = sz
    lib.mla_lowbit_bytes_per_token.argtypes = [lp]
    lib.mla_lowbit_bytes_per_token.restype = sz
    lib.mla_lowbit_write.argtypes = [lp, i32, vp, vp, vp, vp, vp, i32, vp, i32, vp, i64, vp, vp,
                                     vp, vp]
    lib.mla_lowbit_write.restype = i32
    lib.mla_lowbit_decode_plan.argtypes = [lp, i32, i32, vp, i32, ctypes.POINTER(i32),
                                           ctypes.POINTER(i32), ctypes.POINTER(sz)]
    lib.mla_lowbit_decode_plan.restype = i32
    lib.mla_lowbit_decode.argtypes = [lp, i32, i32, ctypes.c_float, vp, vp, i64, vp, i32, vp, vp,
                                      vp, vp, vp, vp, vp, sz, vp, vp]
    lib.mla_lowbit_decode.restype = i32
    lib.mla_lowbit_decode_noalloc.argtypes = [lp, i32, i32, ctypes.c_float, vp, vp, i64, vp, i32,
                                              vp, vp, vp, vp, vp, vp, vp, vp]
    lib.mla_lowbit_decode_noalloc.restype = i32
    lib.mla_lowbit_write_decode.argtypes = [lp, i32, i32, ctypes.c_float, vp, vp, vp, vp, i64, vp,
                                            i32, vp, vp, vp, vp, vp, vp, vp, sz, vp, vp]
    lib.mla_lowbit_write_decode.restype = i32
    lib.mla_lowbit_decode_multi.argtypes = [lp, i32, i32, i32, ctypes.c_float, vp, vp, i64, vp,
                                            i32, vp, vp, vp, vp, vp, vp, vp, sz, vp, vp]
    lib.mla_lowbit_decode_multi.restype = i32
    lib.mla_lowbit_set_fault_injection.argtypes = [i32, i64]
    lib.mla_lowbit_set_fault_injection.restype = i32
    lib.mla_lowbit_read_error.argtypes = [vp, ctypes.POINTER(ctypes.c_int32)]
    lib.mla_lowbit_read_error.restype = i32
    lib.mla_lowbit_strerror.argtypes = [i32]
    lib.mla_lowbit_strerror.restype = ctypes.c_char_p
    lib.mla_lowbit_version.argtypes = []
    lib.mla_lowbit_version.restype = i32
    _LIB = lib
    return lib


def strerror(status: int) -> str:
    return load().mla_lowbit_strerror(int(status)).decode()


def _check(status: int, what: str):
    if status != 0:
        raise LibraryError(f"{what}: {strerror(status)} ({status})")


def page_bytes(lay: Layout) -> int:
    return int(load().mla_lowbit_page_bytes(ctypes.byref(lay)))


def bytes_per_token(lay: Layout) -> int:
    return int(load().mla_lowbit_bytes_per_token(ctypes.byref(lay)))


def version() -> int:
    return int(load().mla_lowbit_version())


def decode_plan(lay: Layout, heads: int, seq_lens_host: Sequence[int], num_sms: int = 0):
    """Returns ``(total_splits, chunk_pages, workspace_bytes)``."""
    lens = np.ascontiguousarray(np.asarray(seq_lens_host, dtype=np.int32))
    tot, chunk, ws = ctypes.c_int(), ctypes.c_int(), ctypes.c_size_t()
    st = load().mla_lowbit_decode_plan(ctypes.byref(lay), len(lens), int(heads),
                                       lens.ctypes.data_as(ctypes.c_void_p), int(num_sms),
                                       ctypes.byref(tot), ctypes.byref(chunk), ctypes.byref(ws))
    _check(st, "mla_lowbit_decode_plan")
    return tot.value, chunk.value, ws.value


# ---------------------------------------------------------------- torch marshalling

def _torch():
    import torch
    return torch


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream, device) -> Optional[int]:
    """The given stream, or the current stream of the device the call runs on."""
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream


def _same_device(device, **tensors):
    """Every CUDA tensor of a call must be on the page pool's device: the
    library launches on the current device, which the call sets to that one."""
    for name, t in tensors.items():
        if t is not None and t.device.type == "cuda" and t.device != device:
            raise ValueError(f"{name} is on {t.device}, the page pool on {device}")


def _expect(t, name, dtype, shape=None, device=True):
    torch = _torch()
    if t is None:
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if device and t.device.type != "cuda":
        raise ValueError(f"{name} must be on a CUDA device")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def write(lay: Layout, ckv, krope, pos, block_table, page_pool, sink_buf, recent_buf, err_word,
          seq_idx=None, seq_lens_after=None, stream=None):
    """Pack ``n`` tokens into the paged cache (mla_lowbit_write)."""
    torch = _torch()
    n = ckv.shape[0]
    _expect(ckv, "ckv", torch.bfloat16, (n, 512))
    _expect(krope, "krope", torch.bfloat16, (n, 64))
    _expect(pos, "pos", torch.int32, (n,))
    _expect(block_table, "block_table", torch.int32)
    _expect(page_pool, "page_pool", torch.uint8)
    _expect(err_word, "err_word", torch.int32, (1,))
    num_seqs, max_pages = block_table.shape
    if seq_idx is not None:
        _expect(seq_idx, "seq_idx", torch.int32, (n,))
    if seq_lens_after is not None:
        _expect(seq_lens_after, "seq_lens_after", torch.int32, (num_seqs,))
    if lay.content_bits != 16:
        _expect(sink_buf, "sink_buf", torch.bfloat16, (num_seqs, 4, 576))
        _expect(recent_buf, "recent_buf", torch.bfloat16, (num_seqs, 128, 576))
    pb = page_bytes(lay)
    if page_pool.dim() != 2 or page_pool.shape[1] != pb:
        raise ValueError(f"page_pool must be [num_pages][{pb}] uint8")
    _same_device(page_pool.device, ckv=ckv, krope=krope, pos=pos, block_table=block_table,
                 sink_buf=sink_buf, recent_buf=recent_buf, err_word=err_word, seq_idx=seq_idx,
                 seq_lens_after=seq_lens_after)
    with torch.cuda.device(page_pool.device):
        st = load().mla_lowbit_write(ctypes.byref(lay), n, _ptr(ckv), _ptr(krope), _ptr(seq_idx),
                                     _ptr(pos), _ptr(seq_lens_after), num_seqs, _ptr(block_table),
                                     max_pages, _ptr(page_pool), page_pool.shape[0], _ptr(sink_buf),
                                     _ptr(recent_buf), _ptr(err_word), _stream(stream, page_pool.device))
    _check(st, "mla_lowbit_write")


def decode(lay: Layout, q, page_pool, block_table, seq_lens, seq_lens_host, sink_buf, recent_buf,
           out, workspace, err_word, softmax_scale: float, lse=None, stream=None):
    """Low-bit MLA decode (mla_lowbit_decode); writes ``out`` (and ``lse``)."""
    torch = _torch()
    B, H, _ = q.shape
    _expect(q, "q", torch.bfloat16, (B, H, 576))
    _expect(page_pool, "page_pool", torch.uint8)
    _expect(block_table, "block_table", torch.int32)
    _expect(seq_lens, "seq_lens", torch.int32, (B,))
    _expect(out, "out", torch.float32, (B, H, 512))
    _expect(workspace, "workspace", torch.uint8)
    _expect(err_word, "err_word", torch.int32, (1,))
    if lse is not None:
        _expect(lse, "lse", torch.float32, (B, H))
    if block_table.shape[0] != B:
        raise ValueError("block_table must have one row per sequence")
    if lay.content_bits != 16:
        _expect(sink_buf, "sink_buf", torch.bfloat16, (B, 4, 576))
        _expect(recent_buf, "recent_buf", torch.bfloat16, (B, 128, 576))
    lens = np.ascontiguousarray(np.asarray(seq_lens_host, dtype=np.int32))
    if lens.shape != (B,):
        raise ValueError("seq_lens_host must have one entry per sequence")
    _same_device(page_pool.device, q=q, block_table=block_table, seq_lens=seq_lens, sink_buf=sink_buf,
                 recent_buf=recent_buf, out=out, workspace=workspace, err_word=err_word, lse=lse)
    with torch.cuda.device(page_pool.device):
        st = load().mla_lowbit_decode(
            ctypes.byref(lay), B, H, ctypes.c_float(softmax_scale), _ptr(q), _ptr(page_pool),
            page_pool.shape[0], _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
            lens.ctypes.data_as(ctypes.c_void_p), _ptr(sink_buf), _ptr(recent_buf), _ptr(out),
            _ptr(lse), _ptr(workspace), workspace.numel(), _ptr(err_word), _stream(stream, page_pool.device))
    _check(st, "mla_lowbit_decode")


def write_decode(lay: Layout, q, ckv_new, krope_new, page_pool, block_table, seq_lens,
                 seq_lens_host, sink_buf, recent_buf, out, workspace, err_word,
                 softmax_scale: float, lse=None, stream=None):
    """mla_lowbit_write_decode: append one token per sequence (at position
    seq_lens[s] - 1) and decode, in one call."""
    torch = _torch()
    B, H, _ = q.shape
    _expect(q, "q", torch.bfloat16, (B, H, 576))
    _expect(ckv_new, "ckv_new", torch.bfloat16, (B, 512))
    _expect(krope_new, "krope_new", torch.bfloat16, (B, 64))
    _expect(page_pool, "page_pool", torch.uint8)
    _expect(block_table, "block_table", torch.int32)
    _expect(seq_lens, "seq_lens", torch.int32, (B,))
    _expect(out, "out", torch.float32, (B, H, 512))
    _expect(workspace, "workspace", torch.uint8)
    _expect(err_word, "err_word", torch.int32, (1,))
    if lse is not None:
        _expect(lse, "lse", torch.float32, (B, H))
    if block_table.shape[0] != B:
        raise ValueError("block_table must have one row per sequence")
    if lay.content_bits != 16:
        _expect(sink_buf, "sink_buf", torch.bfloat16, (B, 4, 576))
        _expect(recent_buf, "recent_buf", torch.bfloat16, (B, 128, 576))
    lens = np.ascontiguousarray(np.asarray(seq_lens_host, dtype=np.int32))
    if lens.shape != (B,):
        raise ValueError("seq_lens_host must have one entry per sequence")
    _same_device(page_pool.device, q=q, ckv_new=ckv_new, krope_new=krope_new, block_table=block_table,
                 seq_lens=seq_lens, sink_buf=sink_buf, recent_buf=recent_buf, out=out,
                 workspace=workspace, err_word=err_word, lse=lse)
    with torch.cuda.device(page_pool.device):
        st = load().mla_lowbit_write_decode(
            ctypes.byref(lay), B, H, ctypes.c_float(softmax_scale), _ptr(q), _ptr(ckv_new),
            _ptr(krope_new), _ptr(page_pool), page_pool.shape[0], _ptr(block_table),
            block_table.shape[1], _ptr(seq_lens), lens.ctypes.data_as(ctypes.c_void_p), _ptr(sink_buf),
            _ptr(recent_buf), _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(),
            _ptr(err_word), _stream(stream, page_pool.device))
    _check(st, "mla_lowbit_write_decode")


def decode_multi(lay: Layout, q, page_pool, block_table, seq_lens, seq_lens_host, sink_buf,
                 recent_buf, out, workspace, err_word, softmax_scale: float, lse=None,
                 stream=None):
    """mla_lowbit_decode_multi: n causal queries per sequence, q [B][n][H][576]."""
    torch = _torch()
    B, n, H, _ = q.shape
    _expect(q, "q", torch.bfloat16, (B, n, H, 576))
    _expect(page_pool, "page_pool", torch.uint8)
    _expect(block_table, "block_table", torch.int32)
    _expect(seq_lens, "seq_lens", torch.int32, (B,))
    _expect(out, "out", torch.float32, (B, n, H, 512))
    _expect(workspace, "workspace", torch.uint8)
    _expect(err_word, "err_word", torch.int32, (1,))
    if lse is not None:
        _expect(lse, "lse", torch.float32, (B, n, H))
    if block_table.shape[0] != B:
        raise ValueError("block_table must have one row per sequence")
    if lay.content_bits != 16:
        _expect(sink_buf, "sink_buf", torch.bfloat16, (B, 4, 576))
        _expect(recent_buf, "recent_buf", torch.bfloat16, (B, 128, 576))
    lens = np.ascontiguousarray(np.asarray(seq_lens_host, dtype=np.int32))
    if lens.shape != (B,):
        raise ValueError("seq_lens_host must have one entry per sequence")
    _same_device(page_pool.device, q=q, block_table=block_table, seq_lens=seq_lens, sink_buf=sink_buf,
                 recent_buf=recent_buf, out=out, workspace=workspace, err_word=err_word, lse=lse)
    with torch.cuda.device(page_pool.device):
        st = load().mla_lowbit_decode_multi(
            ctypes.byref(lay), B, n, H, ctypes.c_float(softmax_scale), _ptr(q), _ptr(page_pool),
            page_pool.shape[0], _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
            lens.ctypes.data_as(ctypes.c_void_p), _ptr(sink_buf), _ptr(recent_buf), _ptr(out),
            _ptr(lse), _ptr(workspace), workspace.numel(), _ptr(err_word), _stream(stream, page_pool.device))
    _check(st, "mla_lowbit_decode_multi")


def decode_noalloc(lay: Layout, q, page_pool, block_table, seq_lens, seq_lens_host, sink_buf,
                   recent_buf, out, err_word, softmax_scale: float, lse=None, stream=None):
    """mla_lowbit_decode_noalloc: the decode without a caller workspace.

    For hosts that can hand the library only inputs and outputs (no device
    allocation allowed); the split partials go to a fixed 32 MiB array the
    library keeps on each device.  Calls that overlap on the GPU race on that
    array, so keep them on one stream."""
    torch = _torch()
    B, H, _ = q.shape
    _expect(q, "q", torch.bfloat16, (B, H, 576))
    _expect(page_pool, "page_pool", torch.uint8)
    _expect(block_table, "block_table", torch.int32)
    _expect(seq_lens, "seq_lens", torch.int32, (B,))
    _expect(out, "out", torch.float32, (B, H, 512))
    _expect(err_word, "err_word", torch.int32, (1,))
    if lse is not None:
        _expect(lse, "lse", torch.float32, (B, H))
    if block_table.shape[0] != B:
        raise ValueError("block_table must have one row per sequence")
    if lay.content_bits != 16:
        _expect(sink_buf, "sink_buf", torch.bfloat16, (B, 4, 576))
        _expect(recent_buf, "recent_buf", torch.bfloat16, (B, 128, 576))
    lens = np.ascontiguousarray(np.asarray(seq_lens_host, dtype=np.int32))
    if lens.shape != (B,):
        raise ValueError("seq_lens_host must have one entry per sequence")
    _same_device(page_pool.device, q=q, block_table=block_table, seq_lens=seq_lens, sink_buf=sink_buf,
                 recent_buf=recent_buf, out=out, err_word=err_word, lse=lse)
    with torch.cuda.device(page_pool.device):
        st = load().mla_lowbit_decode_noalloc(
            ctypes.byref(lay), B, H, ctypes.c_float(softmax_scale), _ptr(q), _ptr(page_pool),
            page_pool.shape[0], _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
            lens.ctypes.data_as(ctypes.c_void_p), _ptr(sink_buf), _ptr(recent_buf), _ptr(out),
            _ptr(lse), _ptr(err_word), _stream(stream, page_pool.device))
    _check(st, "mla_lowbit_decode_noalloc")


def set_fault_injection(mode: int, wait_cycles: int = 0) -> None:
    """Self-test setting of the tcgen05 kernels' bounded waits (process-wide):
    mode 1 withholds one hand-off so that the waits run out after
    ``wait_cycles`` SM cycles (0 = the default limit); mode 0 is normal."""
    _check(load().mla_lowbit_set_fault_injection(int(mode), int(wait_cycles)),
           "mla_lowbit_set_fault_injection")


def read_error(err_word) -> int:
    torch = _torch()
    code = ctypes.c_int32()
    with torch.cuda.device(err_word.device):
        _check(load().mla_lowbit_read_error(_ptr(err_word), ctypes.byref(code)),
               "mla_lowbit_read_error")
    return code.value
