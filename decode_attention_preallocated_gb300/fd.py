"""ctypes binding of libfd.so (the C ABI in include/fd.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels inside libfd.so.  PyTorch supplies device memory and the current
stream.  There is no fallback: if libfd.so is missing or cannot be loaded,
every call raises.

Low-level names mirror the C ABI (``fd_decode``, ``fd_decode_int8``,
``fd_decode_append``, ``fd_decode_paged``, ``fd_decode_masked``,
``fd_decode_gather``, ``fd_decode_gather_int8``, ``fd_decode_gather_bias``,
``fd_topk_blocks``,
``fd_workspace_create`` ...) and take ``FdTensor`` / ``FdOpts`` structures;
``decode``, ``decode_int8``, ``decode_append``, ``decode_paged``,
``decode_masked``, ``decode_gather`` and ``topk_blocks`` take
torch tensors, allocate ``out`` with torch when it is not given, and keep one
workspace per (device, stream).
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfd.so")

# constants from include/fd.h
FD_OK, FD_ERR_ARG, FD_ERR_UNSUPPORTED, FD_ERR_ALIGN, FD_ERR_WORKSPACE, FD_ERR_CUDA = 0, -1, -2, -3, -4, -5
FD_ERR_SCRATCH = -6
FD_BF16, FD_F32, FD_I8, FD_I32 = 0, 1, 2, 3
FD_DEV_BAD_LENGTH, FD_DEV_BAD_INDEX, FD_DEV_INTERNAL = 1, 2, 4
FD_KERNEL_AUTO, FD_KERNEL_SIMT, FD_KERNEL_TC = 0, 1, 2
FD_MAX_ROWS = 64

_DTYPES = {torch.bfloat16: FD_BF16, torch.float32: FD_F32, torch.int8: FD_I8,
           torch.int32: FD_I32}


class FdTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32),
                ("ndim", ctypes.c_int32), ("shape", ctypes.c_int64 * 4),
                ("stride", ctypes.c_int64 * 4)]


class FdOpts(ctypes.Structure):
    _fields_ = [("stream", ctypes.c_void_p), ("ws", ctypes.c_void_p),
                ("num_ctas", ctypes.c_int32), ("kernel", ctypes.c_int32),
                ("scale", ctypes.c_float), ("wait_limit_us", ctypes.c_int32),
                ("reserved", ctypes.c_int32 * 2)]


class FdError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__("%s failed: %s (%d)" % (what, status_string(code), code))


_lib = None
_lib_lock = threading.Lock()

# (name, restype, argtypes) for every symbol declared in include/fd.h
_P = ctypes.POINTER
_SIGNATURES = [
    ("fd_decode", ctypes.c_int,
     [_P(FdTensor), _P(FdTensor), _P(FdTensor), ctypes.c_void_p, ctypes.c_int32,
      ctypes.c_int32, ctypes.c_float, _P(FdTensor), _P(FdOpts)]),
    ("fd_decode_int8", ctypes.c_int,
     [_P(FdTensor), _P(FdTensor), _P(FdTensor), _P(FdTensor), _P(FdTensor),
      ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_float,
      _P(FdTensor), _P(FdOpts)]),
    ("fd_decode_gather", ctypes.c_int,
     [_P(FdTensor), _P(FdTensor), _P(FdTensor), ctypes.c_void_p, ctypes.c_int32,
      _P(FdTensor), _P(FdOpts)]),
    ("fd_decode_gather_int8", ctypes.c_int,
     [_P(FdTensor), _P(FdTensor), _P(FdTensor), _P(FdTensor), _P(FdTensor), ctypes.c_void_p,
      ctypes.c_int32, _P(FdTensor), _P(FdOpts)]),
    ("fd_topk_blocks", ctypes.c_int,
     [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
      ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]),
    ("fd_decode_gather_bias", ctypes.c_int,
     [_P(FdTensor), _P(FdTensor), _P(FdTensor), ctypes.c_void_p, ctypes.c_void_p,
      ctypes.c_int32, _P(FdTensor), _P(FdOpts)]),
    ("fd_decode_masked", ctypes.c_int,
     [_P(FdTensor), _P(FdTensor), _P(FdTensor), ctypes.c_void_p, _P(FdTensor), ctypes.c_int32,
      ctypes.c_int32, ctypes.c_float, _P(FdTensor), _P(FdOpts)]),
    ("fd_decode_append", ctypes.c_int,
     [_P(FdTensor), _P(FdTensor), _P(FdTensor), _P(FdTensor), _P(FdTensor),
      ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_float, _P(FdTensor),
      _P(FdOpts)]),
    ("fd_decode_paged", ctypes.c_int,
     [_P(FdTensor), _P(FdTensor), _P(FdTensor), _P(FdTensor), _P(FdTensor),
      ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
      ctypes.c_float, _P(FdTensor), _P(FdOpts)]),
    ("fd_decode_noalloc", ctypes.c_int,
     [_P(FdTensor), _P(FdTensor), _P(FdTensor), ctypes.c_void_p, ctypes.c_int32,
      ctypes.c_int32, ctypes.c_float, _P(FdTensor), ctypes.c_void_p, ctypes.c_int32]),
    ("fd_workspace_bytes", ctypes.c_size_t,
     [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]),
    ("fd_workspace_create", ctypes.c_int,
     [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
      ctypes.c_void_p, _P(ctypes.c_void_p)]),
    ("fd_workspace_reset", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
    ("fd_workspace_fill_counters", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p]),
    ("fd_workspace_destroy", ctypes.c_int, [ctypes.c_void_p]),
    ("fd_get_device_status", ctypes.c_int, [ctypes.c_void_p, _P(ctypes.c_int32)]),
    ("fd_get_device_diagnostics", ctypes.c_int, [ctypes.c_void_p, _P(ctypes.c_int32)]),
    ("fd_auto_num_ctas", ctypes.c_int32,
     [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64]),
    ("fd_tile_tokens", ctypes.c_int32, [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]),
    ("fd_masked_list_bytes", ctypes.c_size_t, [ctypes.c_int64, ctypes.c_int64]),
    ("fd_plan", ctypes.c_int64,
     [_P(ctypes.c_int64), ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
      _P(ctypes.c_int32), _P(ctypes.c_int32)]),
    ("fd_seg_units", ctypes.c_int32, [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]),
    ("fd_status_string", ctypes.c_char_p, [ctypes.c_int]),
    ("fd_version", ctypes.c_int32, []),
]


def lib() -> ctypes.CDLL:
    """Load libfd.so (raises if it has not been built)."""
    global _lib
    with _lib_lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    "libfd.so is not built (%s); run "
                    "decode_attention_preallocated_gb300.build.build()" % LIB_PATH)
            h = ctypes.CDLL(LIB_PATH)
            for name, res, args in _SIGNATURES:
                fn = getattr(h, name)
                fn.restype = res
                fn.argtypes = args
            _lib = h
    return _lib


def status_string(code: int) -> str:
    return lib().fd_status_string(int(code)).decode()


# ------------------------------------------------------------- marshalling
def as_fd_tensor(t: torch.Tensor) -> FdTensor:
    dt = _DTYPES.get(t.dtype)
    if dt is None:
        raise TypeError("unsupported dtype %s" % t.dtype)
    shape = t.shape
    n = len(shape)
    if n > 4:
        raise ValueError("at most 4 dimensions")
    ft = FdTensor()
    ft.data = t.data_ptr()
    ft.dtype = dt
    ft.ndim = n
    ft.shape[:n] = shape
    ft.stride[:n] = t.stride()
    return ft


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_handle(stream: Optional[torch.cuda.Stream], device) -> int:
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None:
        return _raw_stream(device.index)
    return torch.cuda.current_stream(device).cuda_stream


class _on_device:
    """Makes `device` current for the C call, unless it already is."""

    __slots__ = ("device", "prev")

    def __init__(self, device):
        self.device = device
        self.prev = None

    def __enter__(self):
        cur = torch.cuda.current_device()
        if cur != self.device.index:
            self.prev = cur
            torch.cuda.set_device(self.device)

    def __exit__(self, *exc):
        if self.prev is not None:
            torch.cuda.set_device(self.prev)
        return False


def _check(code: int, what: str):
    if code != FD_OK:
        raise FdError(code, what)


# -------------------------------------------------------------- workspace
class Workspace:
    """Owns one fd_workspace (device memory allocated by libfd.so).

    Size it for the largest call it will serve; a call that needs more fails
    with FD_ERR_WORKSPACE.  Create it before capturing a CUDA graph.
    """

    def __init__(self, max_segments: int, max_rows: int, head_dim: int,
                 max_ctas: int, stream: Optional[torch.cuda.Stream] = None,
                 device=None):
        self.max_segments, self.max_rows = int(max_segments), int(max_rows)
        self.head_dim, self.max_ctas = int(head_dim), int(max_ctas)
        self.device = torch.device("cuda", torch.cuda.current_device()) \
            if device is None else torch.device(device)
        h = ctypes.c_void_p()
        with torch.cuda.device(self.device):
            _check(lib().fd_workspace_create(self.max_segments, self.max_rows,
                                             self.head_dim, self.max_ctas,
                                             _stream_handle(stream, self.device),
                                             ctypes.byref(h)),
                   "fd_workspace_create")
        self.handle = h

    def fits(self, segments, rows, head_dim, ctas) -> bool:
        return (segments <= self.max_segments and rows <= self.max_rows
                and head_dim <= self.head_dim and ctas <= self.max_ctas)

    def reset(self, stream=None):
        _check(lib().fd_workspace_reset(self.handle, _stream_handle(stream, self.device)),
               "fd_workspace_reset")

    def fill_counters(self, value: int, stream=None):
        """Test hook: every completion counter set to `value` (a negative one
        stands for counters an aborted launch left behind)."""
        _check(lib().fd_workspace_fill_counters(self.handle, int(value),
                                                _stream_handle(stream, self.device)),
               "fd_workspace_fill_counters")

    def device_status(self) -> int:
        st = ctypes.c_int32(0)
        with torch.cuda.device(self.device):
            _check(lib().fd_get_device_status(self.handle, ctypes.byref(st)),
                   "fd_get_device_status")
        return int(st.value)

    def diagnostics(self):
        w = (ctypes.c_int32 * 13)()
        with torch.cuda.device(self.device):
            _check(lib().fd_get_device_diagnostics(self.handle, w), "fd_get_device_diagnostics")
        return list(w)

    def close(self):
        if getattr(self, "handle", None) is not None and self.handle.value:
            with torch.cuda.device(self.device):
                torch.cuda.synchronize(self.device)
                lib().fd_workspace_destroy(self.handle)
            self.handle = None

    def __del__(self):  # pragma: no cover - best effort at interpreter exit
        try:
            self.close()
        except Exception:
            pass


_ws_cache = {}
_ws_lock = threading.Lock()


def workspace_for(device, stream_handle, segments, rows, head_dim, ctas) -> Workspace:
    """Workspace shared by calls on one (device, stream); grown when needed
    (growth synchronises the device, so size it up front for graph capture)."""
    key = (torch.device(device).index, int(stream_handle))
    with _ws_lock:
        ws = _ws_cache.get(key)
        if ws is None or not ws.fits(segments, rows, head_dim, ctas):
            want = dict(max_segments=max(segments, 64), max_rows=max(rows, 16),
                        head_dim=max(head_dim, 256), max_ctas=max(ctas, 1024))
            if ws is not None:
                want = dict(max_segments=max(want["max_segments"], ws.max_segments),
                            max_rows=max(want["max_rows"], ws.max_rows),
                            head_dim=max(want["head_dim"], ws.head_dim),
                            max_ctas=max(want["max_ctas"], ws.max_ctas))
                ws.close()
            ws = Workspace(device=device, **want)
            _ws_cache[key] = ws
        return ws


def auto_num_ctas(kernel=FD_KERNEL_AUTO, head_dim=128, kv_dtype=FD_BF16, rows=1,
                  max_tiles=0) -> int:
    return int(lib().fd_auto_num_ctas(kernel, head_dim, kv_dtype, rows, max_tiles))


def tile_tokens(kernel=FD_KERNEL_AUTO, head_dim=128, kv_dtype=FD_BF16) -> int:
    return int(lib().fd_tile_tokens(kernel, head_dim, kv_dtype))


def masked_list_bytes(B, cap) -> int:
    """Workspace bytes, past a masked call's split partials, that let the
    tensor-core kernel list the visible chunks before it decodes."""
    return int(lib().fd_masked_list_bytes(int(B), int(cap)))


def slot_floats(rows, head_dim) -> int:
    """Floats of one workspace slot of split partials (O, m and l of rows)."""
    return rows * head_dim + ((2 * rows + 3) // 4) * 4


def plan(seg_len, tile, num_ctas, seg_units=0):
    """Host mirror of the device partitioner: (total work units, first block
    of each segment, number of blocks sharing each segment).  Each non-empty
    segment is charged `seg_units` units before its tiles."""
    n = len(seg_len)
    arr = (ctypes.c_int64 * max(n, 1))(*[int(x) for x in seg_len])
    first = (ctypes.c_int32 * max(n, 1))()
    pieces = (ctypes.c_int32 * max(n, 1))()
    total = lib().fd_plan(arr, n, int(tile), int(num_ctas), int(seg_units), first, pieces)
    if total < 0:
        raise FdError(int(total), "fd_plan")
    return int(total), list(first)[:n], list(pieces)[:n]


def seg_units(kernel, head_dim, kv_dtype=FD_BF16):
    """Work units a launch of `kernel` charges per segment start."""
    return int(lib().fd_seg_units(int(kernel), int(head_dim), int(kv_dtype)))


# ---------------------------------------------------------- torch wrappers
def _opts(stream_handle, ws, num_ctas, kernel, scale=0.0, wait_limit_us=0) -> FdOpts:
    o = FdOpts()
    o.stream = stream_handle
    o.ws = ws.handle
    o.num_ctas = int(num_ctas)
    o.kernel = int(kernel)
    o.scale = float(scale)
    o.wait_limit_us = int(wait_limit_us)
    return o


def _prepare(q, k, out, out_dtype, segments, rows, num_ctas, kernel, stream, ws):
    if not q.is_cuda:
        raise ValueError("q must be a CUDA tensor")
    device = q.device
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype, device=device)
    sh = _stream_handle(stream, device)
    if ws is None:
        ctas = num_ctas
        if ctas == 0:
            # an upper bound on what either kernel picks for an auto launch
            with torch.cuda.device(device):
                ctas = max(auto_num_ctas(FD_KERNEL_SIMT, q.shape[-1], FD_BF16, rows, 0),
                           auto_num_ctas(FD_KERNEL_TC, q.shape[-1], FD_BF16, rows, 0))
        ws = workspace_for(device, sh, segments, rows, q.shape[-1], max(ctas, 1))
    return out, sh, ws


def decode(q, k_cache, v_cache, kv_lengths, n_q=None, causal=False, scale=None,
           out=None, out_dtype=torch.bfloat16, num_ctas=0, kernel=FD_KERNEL_AUTO,
           stream=None, workspace: Optional[Workspace] = None, wait_limit_us=0):
    """Attention of q [B, n_q, Hq, d] over the first kv_lengths[b] positions of
    k_cache / v_cache [B, Hkv, cap, d] (bf16).  kv_lengths: int32 [B] on the
    device.  Returns out [B, n_q, Hq, d].  wait_limit_us bounds each internal
    wait of the tensor-core kernel (0: 2 s)."""
    B, nq, Hq, d = q.shape
    n_q = nq if n_q is None else n_q
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    Hkv = k_cache.shape[1]
    rows = (Hq // max(Hkv, 1)) * nq
    out, sh, ws = _prepare(q, k_cache, out, out_dtype, B * Hkv, rows, num_ctas,
                           kernel, stream, workspace)
    tq, tk, tv, to = map(as_fd_tensor, (q, k_cache, v_cache, out))
    o = _opts(sh, ws, num_ctas, kernel, wait_limit_us=wait_limit_us)
    with _on_device(q.device):
        rc = lib().fd_decode(ctypes.byref(tq), ctypes.byref(tk), ctypes.byref(tv),
                             kv_lengths.data_ptr(), int(n_q), int(bool(causal)),
                             float(scale), ctypes.byref(to), ctypes.byref(o))
    _check(rc, "fd_decode")
    return out


def decode_int8(q, k_cache, v_cache, k_scale, v_scale, kv_lengths, n_q=None,
                causal=False, scale=None, out=None, out_dtype=torch.bfloat16,
                num_ctas=0, kernel=FD_KERNEL_AUTO, stream=None,
                workspace: Optional[Workspace] = None):
    """As ``decode`` for an int8 cache with fp32 scales [B, Hkv, cap]."""
    B, nq, Hq, d = q.shape
    n_q = nq if n_q is None else n_q
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    Hkv = k_cache.shape[1]
    rows = (Hq // max(Hkv, 1)) * nq
    # more than 32 rows: the tensor-core kernel serves each kv head's query
    # heads in parts, a segment each (at most one per query head)
    segments = B * Hq if rows > 32 else B * Hkv
    out, sh, ws = _prepare(q, k_cache, out, out_dtype, segments, rows, num_ctas,
                           kernel, stream, workspace)
    tq, tk, tv, tks, tvs, to = map(as_fd_tensor, (q, k_cache, v_cache, k_scale, v_scale, out))
    o = _opts(sh, ws, num_ctas, kernel)
    with _on_device(q.device):
        rc = lib().fd_decode_int8(ctypes.byref(tq), ctypes.byref(tk), ctypes.byref(tv),
                                  ctypes.byref(tks), ctypes.byref(tvs),
                                  kv_lengths.data_ptr(), int(n_q), int(bool(causal)),
                                  float(scale), ctypes.byref(to), ctypes.byref(o))
    _check(rc, "fd_decode_int8")
    return out


def topk_blocks(scores, kv_lengths, block_size, top_k, out=None, stream=None):
    """Gather lists from block scores: scores fp32 [B, n_q, n_blocks]
    (contiguous, on the device), kv_lengths int32 [B].  Returns (or fills)
    idx int32 [B, n_q, top_k*block_size]: the top_k blocks of each row in
    increasing order, expanded to cells, -1 past the length or unused."""
    if not scores.is_cuda or scores.dtype != torch.float32 or scores.dim() != 3 \
            or not scores.is_contiguous():
        raise ValueError("scores must be a contiguous CUDA float32 [B, n_q, n_blocks] tensor")
    B, n_q, nb = scores.shape
    W = int(top_k) * int(block_size)
    if out is None:
        out = torch.empty((B, n_q, W), dtype=torch.int32, device=scores.device)
    sh = _stream_handle(stream, scores.device)
    with _on_device(scores.device):
        rc = lib().fd_topk_blocks(scores.data_ptr(), B, n_q, nb, kv_lengths.data_ptr(),
                                  int(block_size), int(top_k), out.data_ptr(), sh)
    _check(rc, "fd_topk_blocks")
    return out


def decode_masked(q, k_cache, v_cache, kv_lengths, mask, n_q=None, causal=False, scale=None,
                  out=None, out_dtype=torch.bfloat16, num_ctas=0, kernel=FD_KERNEL_AUTO,
                  stream=None, workspace: Optional[Workspace] = None):
    """As ``decode`` with an additive fp32 mask [B, n_q, cap] (positions
    contiguous; -inf hides a position); 32-position chunks the mask hides for
    every query row are not read.  The default workspace leaves room for the
    tensor-core kernel's chunk list (its time then follows the visible
    chunks)."""
    B, nq, Hq, d = q.shape
    n_q = nq if n_q is None else n_q
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    Hkv = k_cache.shape[1]
    rows = (Hq // max(Hkv, 1)) * nq
    # room for the chunk list, counted in slots of the call's partials
    extra = -(-masked_list_bytes(B, k_cache.shape[2]) // (4 * slot_floats(rows, d)))
    out, sh, ws = _prepare(q, k_cache, out, out_dtype, B * Hkv + extra, rows, num_ctas,
                           kernel, stream, workspace)
    tq, tk, tv, tm, to = map(as_fd_tensor, (q, k_cache, v_cache, mask, out))
    o = _opts(sh, ws, num_ctas, kernel)
    with _on_device(q.device):
        rc = lib().fd_decode_masked(ctypes.byref(tq), ctypes.byref(tk), ctypes.byref(tv),
                                    kv_lengths.data_ptr(), ctypes.byref(tm), int(n_q),
                                    int(bool(causal)), float(scale), ctypes.byref(to),
                                    ctypes.byref(o))
    _check(rc, "fd_decode_masked")
    return out


def decode_append(q, k_cache, v_cache, k_new, v_new, kv_lengths, causal=True, scale=None,
                  update_lengths=True, out=None, out_dtype=torch.bfloat16, num_ctas=0,
                  kernel=FD_KERNEL_AUTO, stream=None, workspace: Optional[Workspace] = None):
    """One decode step with a fused append: writes k_new / v_new
    [B, n_q, Hkv, d] (bf16) into k_cache / v_cache [B, Hkv, cap, d] at
    positions kv_lengths[b] .. kv_lengths[b] + n_q - 1, attends q
    [B, n_q, Hq, d] over the prefix including them (row i sees up to
    kv_lengths[b] + i when causal) and, with update_lengths, advances
    kv_lengths (int32 [B], on the device) by n_q when the launch ends."""
    B, nq, Hq, d = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    Hkv = k_cache.shape[1]
    rows = (Hq // max(Hkv, 1)) * nq
    out, sh, ws = _prepare(q, k_cache, out, out_dtype, B * Hkv, rows, num_ctas,
                           kernel, stream, workspace)
    tq, tk, tv, tkn, tvn, to = map(as_fd_tensor, (q, k_cache, v_cache, k_new, v_new, out))
    o = _opts(sh, ws, num_ctas, kernel)
    with _on_device(q.device):
        rc = lib().fd_decode_append(ctypes.byref(tq), ctypes.byref(tk), ctypes.byref(tv),
                                    ctypes.byref(tkn), ctypes.byref(tvn), kv_lengths.data_ptr(),
                                    int(bool(update_lengths)), int(bool(causal)), float(scale),
                                    ctypes.byref(to), ctypes.byref(o))
    _check(rc, "fd_decode_append")
    return out


def decode_paged(q, k_pages, v_pages, block_table, kv_lengths, n_q=None,
                 causal=False, scale=None, k_scale=None, v_scale=None, out=None,
                 out_dtype=torch.bfloat16, num_ctas=0, kernel=FD_KERNEL_AUTO,
                 stream=None, workspace: Optional[Workspace] = None):
    """As ``decode`` (or ``decode_int8``) over a paged cache: pools
    k_pages / v_pages [num_pages, Hkv, page_size, d] (bf16, or int8 with fp32
    scales [num_pages, Hkv, page_size]) and block_table [B, max_pages] (int32,
    contiguous, on the device): position j of sequence b is row
    j % page_size of page block_table[b, j // page_size]."""
    B, nq, Hq, d = q.shape
    n_q = nq if n_q is None else n_q
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    if (not block_table.is_contiguous() or block_table.dtype != torch.int32
            or block_table.dim() != 2 or block_table.shape[0] != B):
        raise ValueError("block_table must be a contiguous int32 [B, max_pages] tensor")
    Hkv = k_pages.shape[1]
    rows = (Hq // max(Hkv, 1)) * nq
    out, sh, ws = _prepare(q, k_pages, out, out_dtype, B * Hkv, rows, num_ctas,
                           kernel, stream, workspace)
    tq, tk, tv, to = map(as_fd_tensor, (q, k_pages, v_pages, out))
    pks = pvs = None
    if k_scale is not None or v_scale is not None:
        tks, tvs = as_fd_tensor(k_scale), as_fd_tensor(v_scale)
        pks, pvs = ctypes.byref(tks), ctypes.byref(tvs)
    o = _opts(sh, ws, num_ctas, kernel)
    with _on_device(q.device):
        rc = lib().fd_decode_paged(ctypes.byref(tq), ctypes.byref(tk), ctypes.byref(tv),
                                   pks, pvs, block_table.data_ptr(), int(block_table.shape[1]),
                                   kv_lengths.data_ptr(), int(n_q), int(bool(causal)),
                                   float(scale), ctypes.byref(to), ctypes.byref(o))
    _check(rc, "fd_decode_paged")
    return out


def decode_gather(q, k_cache, v_cache, idx, scale=None, out=None,
                  out_dtype=torch.bfloat16, num_ctas=0, kernel=FD_KERNEL_AUTO,
                  stream=None, workspace: Optional[Workspace] = None, bias=None,
                  k_scale=None, v_scale=None):
    """Attention of q [B, n_q, Hq, d] over the cache cells listed in
    idx [B, n_q, K] (int32, contiguous, on the device; < 0 = padding).
    bias (optional, bf16 caches): fp32 [B, n_q, K] contiguous, added to each
    entry's score (-inf drops the entry).  int8 caches take fp32 k_scale /
    v_scale [B, Hkv, cap] (fd_decode_gather_int8)."""
    B, nq, Hq, d = q.shape
    Hkv = k_cache.shape[1]
    if not idx.is_contiguous() or idx.dtype != torch.int32 or idx.dim() != 3:
        raise ValueError("idx must be a contiguous int32 [B, n_q, K] tensor")
    rows = Hq // max(Hkv, 1)
    out, sh, ws = _prepare(q, k_cache, out, out_dtype, B * nq * Hkv, rows, num_ctas,
                           kernel, stream, workspace)
    tq, tk, tv, to = map(as_fd_tensor, (q, k_cache, v_cache, out))
    o = _opts(sh, ws, num_ctas, kernel, 0.0 if scale is None else scale)
    if k_cache.dtype == torch.int8:
        if bias is not None or k_scale is None or v_scale is None:
            raise ValueError("int8 caches take k_scale and v_scale, and no bias")
        tks, tvs = as_fd_tensor(k_scale), as_fd_tensor(v_scale)
        with _on_device(q.device):
            rc = lib().fd_decode_gather_int8(ctypes.byref(tq), ctypes.byref(tk), ctypes.byref(tv),
                                             ctypes.byref(tks), ctypes.byref(tvs), idx.data_ptr(),
                                             int(idx.shape[2]), ctypes.byref(to), ctypes.byref(o))
        _check(rc, "fd_decode_gather_int8")
        return out
    if bias is not None:
        if (not bias.is_contiguous() or bias.dtype != torch.float32
                or tuple(bias.shape) != tuple(idx.shape)):
            raise ValueError("bias must be a contiguous float32 tensor shaped like idx")
        with _on_device(q.device):
            rc = lib().fd_decode_gather_bias(ctypes.byref(tq), ctypes.byref(tk),
                                             ctypes.byref(tv), idx.data_ptr(), bias.data_ptr(),
                                             int(idx.shape[2]), ctypes.byref(to),
                                             ctypes.byref(o))
        _check(rc, "fd_decode_gather_bias")
        return out
    with _on_device(q.device):
        rc = lib().fd_decode_gather(ctypes.byref(tq), ctypes.byref(tk), ctypes.byref(tv),
                                    idx.data_ptr(), int(idx.shape[2]), ctypes.byref(to),
                                    ctypes.byref(o))
    _check(rc, "fd_decode_gather")
    return out
