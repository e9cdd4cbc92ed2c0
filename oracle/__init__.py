"""fp64 CPU oracle for length-aware GQA decode attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the benchmark's CPU-baseline leg may import this package.  The product path
(``decode_attention_preallocated_gb300``) never imports it, and it never
imports the product path: the two share no code.  Inputs reach both sides
from ``decode_attention_preallocated_gb300.workloads`` (seeded generators
only, no attention arithmetic).

``dense`` and ``gather`` call the plain C loops in ``fd_oracle.c``
(definition in that file's header); ``bruteforce`` is a second, pure-Python
path used to pin the C code on tiny inputs.

Parity pins (each checked by ``tests/test_oracle_pins.py``):
  * closed forms: one visible key returns its value row; identical keys
    return the mean of the visible value rows; constant values are returned
    unchanged; q = 0 gives the uniform mean; a dominant key returns its row;
  * library special case: ``torch.nn.functional.scaled_dot_product_attention``
    in float64 with an explicit boolean mask and repeated KV heads;
  * brute force: ``oracle.bruteforce`` (math.fsum over Python floats);
  * invariants: gather over 0..L-1 equals the dense prefix, gather over a
    selection equals the masked dense path, permutation invariance of the
    gather list, independence from capacity beyond the length and from the
    tail contents, causal row i ignores drafts after i, length rollback;
  * hand-derived closed-form fixtures under ``tests/golden``.
The pages print no attention values for a worked example, so no pin comes
from printed numbers.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fd_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``fd_oracle.c`` into ``liboracle.so`` (gcc, OpenMP, -O2)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c99",
           "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(path):
    lib = ctypes.CDLL(path)
    p = ctypes.c_void_p
    i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
    lib.fdo_dense.argtypes = [p, p, p, p, p, p, i32, p, p, p, p,
                              i32, i32, i32, i32, i32, i64, i32, f64, p]
    lib.fdo_dense.restype = i32
    lib.fdo_gather.argtypes = [p, p, p, p, p, p, i32, p, p, p, p, i64,
                               i32, i32, i32, i32, i32, i64, f64, p]
    lib.fdo_gather.restype = i32
    lib.fdo_gather_bias.argtypes = [p, p, p, p, p, p, i32, p, p, p, p, p, i64,
                                    i32, i32, i32, i32, i32, i64, f64, p]
    lib.fdo_gather_bias.restype = i32
    lib.fdo_set_threads.argtypes = [i32]
    lib.fdo_set_threads.restype = None
    lib.fdo_max_threads.argtypes = []
    lib.fdo_max_threads.restype = i32
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = _bind(_LIB_PATH)
    return _lib


def load_variant(path: str):
    """Bind another build of ``fd_oracle.c`` (used by the mutation tests that
    plant mistakes in copies of the oracle).  Returns an object with the same
    ``dense`` / ``gather`` functions as this module."""
    lib = _bind(path)

    class _Variant:
        @staticmethod
        def dense(*a, **kw):
            return dense(*a, _lib_override=lib, **kw)

        @staticmethod
        def gather(*a, **kw):
            return gather(*a, _lib_override=lib, **kw)

    return _Variant


def set_threads(n: int) -> None:
    _load().fdo_set_threads(int(n))


def max_threads() -> int:
    return int(_load().fdo_max_threads())


def _as_np(t):
    """torch CPU tensor or numpy array -> (numpy array, element strides).

    bf16 tensors are reinterpreted as their uint16 bit patterns; the oracle
    widens them exactly.  Strides are kept, so strided views work.
    """
    try:
        import torch
    except ImportError:  # pragma: no cover
        torch = None
    if torch is not None and isinstance(t, torch.Tensor):
        t = t.detach()
        if t.device.type != "cpu":
            t = t.cpu()
        if t.dtype == torch.bfloat16:
            base = t.view(torch.int16)
            arr = base.numpy().view(np.uint16)
        else:
            arr = t.numpy()
        return arr
    return np.asarray(t)


def _strides(arr):
    return np.asarray([s // arr.itemsize for s in arr.strides], dtype=np.int64)


def _ptr(arr):
    return arr.ctypes.data_as(ctypes.c_void_p)


def _kv_args(k, v, k_scale, v_scale):
    ka, va = _as_np(k), _as_np(v)
    if ka.dtype == np.int8:
        if k_scale is None or v_scale is None:
            raise ValueError("int8 caches need k_scale and v_scale")
        ks_a = np.asarray(_as_np(k_scale), dtype=np.float32)
        vs_a = np.asarray(_as_np(v_scale), dtype=np.float32)
        if _strides(ks_a).tolist() != _strides(vs_a).tolist():
            vs_a = np.ascontiguousarray(vs_a)
            ks_a = np.ascontiguousarray(ks_a)
        int8 = 1
    elif ka.dtype == np.uint16:
        ks_a = vs_a = None
        int8 = 0
    else:
        raise TypeError("k/v must be bf16 or int8, got %s" % ka.dtype)
    if va.dtype != ka.dtype:
        raise TypeError("k and v must have the same dtype")
    return ka, va, ks_a, vs_a, int8


def dense(q, k, v, kv_lengths, n_q, causal, scale, k_scale=None,
          v_scale=None, _lib_override=None):
    """fp64 attention over the filled prefix (optionally bottom-right causal).

    q [B, n_q, Hq, d] bf16; k, v [B, Hkv, cap, d] bf16 or int8 (any strides);
    kv_lengths [B] int32 host values; int8 caches take fp32 scales
    [B, Hkv, cap].  Returns float64 [B, n_q, Hq, d].
    """
    lib = _lib_override or _load()
    qa = _as_np(q)
    if qa.dtype != np.uint16:
        raise TypeError("q must be bf16")
    ka, va, ksa, vsa, int8 = _kv_args(k, v, k_scale, v_scale)
    B, nq_, Hq, d = qa.shape
    if nq_ != n_q:
        raise ValueError("q.shape[1] != n_q")
    _, Hkv, cap, d2 = ka.shape
    if d2 != d or va.shape != ka.shape:
        raise ValueError("shape mismatch")
    lens = np.ascontiguousarray(np.asarray(_as_np(kv_lengths), dtype=np.int32))
    if lens.shape != (B,):
        raise ValueError("kv_lengths must be [B]")
    out = np.zeros((B, n_q, Hq, d), dtype=np.float64)
    qs, ks, vs = _strides(qa), _strides(ka), _strides(va)
    ss = _strides(ksa) if int8 else np.zeros(3, dtype=np.int64)
    rc = lib.fdo_dense(_ptr(qa), _ptr(qs), _ptr(ka), _ptr(ks), _ptr(va),
                       _ptr(vs), int8,
                       _ptr(ksa) if int8 else None,
                       _ptr(vsa) if int8 else None, _ptr(ss), _ptr(lens),
                       B, n_q, Hq, Hkv, d, cap, 1 if causal else 0,
                       float(scale), _ptr(out))
    if rc != 0:
        raise RuntimeError("fdo_dense failed: %d" % rc)
    return out


def masked(q, k, v, kv_lengths, mask, n_q, causal, scale):
    """fp64 attention over the filled prefix with an additive mask
    ("qwen4exp : gather-based sparse attention for QSA decode", llama.cpp
    #28213: the selection as a mask over the window; the Metal FA-vec kernel
    skips the chunks it hides).

    The visible positions of row (b, i) are those of ``dense`` whose
    mask[b, i, j] is not -inf; each one's score gains mask[b, i, j].  The
    positions and mask values are handed to ``gather`` as the row's list and
    per-entry bias.  mask: fp32 [B, n_q, cap].  Returns float64
    [B, n_q, Hq, d].
    """
    qa = _as_np(q)
    ma = np.asarray(_as_np(mask), dtype=np.float32)
    B = qa.shape[0]
    cap = _as_np(k).shape[2]
    if ma.shape != (B, n_q, cap):
        raise ValueError("mask must be [B, n_q, cap]")
    lens = np.clip(np.asarray(_as_np(kv_lengths), dtype=np.int64).reshape(B), 0, cap)
    rows = []
    for b in range(B):
        L = int(lens[b])
        for i in range(n_q):
            last = L - n_q + i if causal else L - 1
            cells = np.arange(max(0, min(L, last + 1)))
            cells = cells[ma[b, i, cells] != -np.inf]
            rows.append(cells)
    K = max(1, max(len(r) for r in rows))
    idx = np.full((B * n_q, K), -1, dtype=np.int32)
    bias = np.zeros((B * n_q, K), dtype=np.float32)
    for r, cells in enumerate(rows):
        idx[r, :len(cells)] = cells
        bias[r, :len(cells)] = ma[r // n_q, r % n_q, cells]
    return gather(qa, k, v, idx.reshape(B, n_q, K), scale, bias=bias.reshape(B, n_q, K))


def topk_blocks(scores, kv_lengths, block_size, top_k):
    """Index lists from block scores: top-k over blocks, then only the
    winners expanded to cells ("qwen4exp : gather-based sparse attention for
    QSA decode", llama.cpp #28213, review discussion: take top-k over blocks
    and expand only the winners).

    scores: fp32 [B, n_q, n_blocks], block j covering cells
    j*block_size .. (j+1)*block_size - 1; kv_lengths [B] (host).  For row
    (b, i), with L = kv_lengths[b] clamped to [0, n_blocks*block_size], the
    candidates are the blocks whose first cell is below L; the top_k highest
    scores win, ties going to the lower block index.  The winners are listed
    in increasing block order, each expanded to its block_size cells, cells
    at or past L written as -1, and the list padded with -1 to
    top_k*block_size entries.  Returns int32 [B, n_q, top_k*block_size].
    """
    sc = np.asarray(_as_np(scores), dtype=np.float32)
    B, n_q, nb = sc.shape
    lens = np.asarray(_as_np(kv_lengths), dtype=np.int64).reshape(B)
    W = top_k * block_size
    out = np.full((B, n_q, W), -1, dtype=np.int32)
    for b in range(B):
        L = int(min(max(lens[b], 0), nb * block_size))
        nvalid = min(nb, -(-L // block_size))
        cand = np.arange(nvalid)
        for i in range(n_q):
            s = sc[b, i, :nvalid].astype(np.float64)
            # sort by score descending, then block index ascending
            order = np.lexsort((cand, -s))
            chosen = np.sort(order[:top_k])
            cells = (chosen[:, None] * block_size + np.arange(block_size)[None, :]).ravel()
            cells = np.where(cells < L, cells, -1)
            out[b, i, :cells.size] = cells
    return out


def append(q, k, v, k_new, v_new, kv_lengths, causal, scale):
    """One decode step with an append, as flash_attn_with_kvcache defines it
    (ComfyUI #16509, Existing Solutions): the new rows go into the cache at
    each sequence's length, then ``dense`` attends over the longer prefix.

    q [B, n, Hq, d] bf16 (the n new tokens); k, v [B, Hkv, cap, d] bf16;
    k_new, v_new [B, n, Hkv, d] bf16; kv_lengths [B] host int32 (lengths
    before the step).  With base_b = clamp(kv_lengths[b], 0, cap), row i of
    sequence b is written at position base_b + i when that is below cap, and
    the step's length is min(base_b + n, cap).  Returns (out float64
    [B, n, Hq, d], k after, v after (uint16 bf16 bits, the inputs are not
    modified), lengths after int32 [B]).
    """
    qa = _as_np(q)
    ka = np.array(_as_np(k), copy=True)
    va = np.array(_as_np(v), copy=True)
    kn, vn = _as_np(k_new), _as_np(v_new)
    B, n, Hq, d = qa.shape
    _, Hkv, cap, _ = ka.shape
    if kn.shape != (B, n, Hkv, d) or vn.shape != kn.shape:
        raise ValueError("k_new / v_new must be [B, n_q, Hkv, d]")
    lens = np.asarray(_as_np(kv_lengths), dtype=np.int64).reshape(B)
    base = np.clip(lens, 0, cap)
    for b in range(B):
        for i in range(n):
            pos = int(base[b]) + i
            if pos < cap:
                ka[b, :, pos, :] = kn[b, i]
                va[b, :, pos, :] = vn[b, i]
    after = np.minimum(base + n, cap).astype(np.int32)
    out = dense(qa, ka, va, after, n, causal, scale)
    return out, ka, va, after


def paged(q, k_pages, v_pages, block_table, kv_lengths, n_q, causal, scale,
          k_scale=None, v_scale=None, _lib_override=None):
    """fp64 attention over a paged cache: the dense prefix definition with
    one indirection (comfy-kitchen #239, commit list and Description: a
    bounded paged int8 decode cache with rollback).

    Position j of sequence b is row j % page_size of pool page
    block_table[b, j // page_size].  Pools k_pages, v_pages are
    [num_pages, Hkv, page_size, d] (bf16, or int8 with fp32 scales
    [num_pages, Hkv, page_size]); block_table [B, max_pages] int32 and
    kv_lengths [B] int32 are host values.  The visible positions of query
    row i are those of ``dense`` -- j < L_b with L_b clamped to
    [0, max_pages * page_size], and j <= L_b - n_q + i for causal windows --
    minus the positions on a page whose table entry is outside
    [0, num_pages).

    Each sequence's logical cache is assembled row by row from the pool,
    and each (sequence, query row)'s visible positions are handed to
    ``gather`` as its list.  Returns float64 [B, n_q, Hq, d].
    """
    qa = _as_np(q)
    ka, va, ksa, vsa, int8 = _kv_args(k_pages, v_pages, k_scale, v_scale)
    B, nq_, Hq, d = qa.shape
    if nq_ != n_q:
        raise ValueError("q.shape[1] != n_q")
    P, Hkv, ps, d2 = ka.shape
    if d2 != d or va.shape != ka.shape:
        raise ValueError("shape mismatch")
    table = np.asarray(_as_np(block_table), dtype=np.int64)
    if table.ndim != 2 or table.shape[0] != B:
        raise ValueError("block_table must be [B, max_pages]")
    max_pages = table.shape[1]
    cap = max_pages * ps
    lens = np.clip(np.asarray(_as_np(kv_lengths), dtype=np.int64).reshape(B), 0, cap)
    # logical caches [B, Hkv, cap, d]: position j <- pool[page(j), :, j % ps, :]
    j = np.arange(cap)
    page = table[:, j // ps]                      # [B, cap]
    on_pool = (page >= 0) & (page < P)
    pg = np.where(on_pool, page, 0)
    row = np.broadcast_to(j % ps, pg.shape)
    k_log = np.ascontiguousarray(np.transpose(ka[pg, :, row, :], (0, 2, 1, 3)))
    v_log = np.ascontiguousarray(np.transpose(va[pg, :, row, :], (0, 2, 1, 3)))
    ks_log = vs_log = None
    if int8:
        ks_log = np.ascontiguousarray(np.transpose(ksa[pg, :, row], (0, 2, 1)))
        vs_log = np.ascontiguousarray(np.transpose(vsa[pg, :, row], (0, 2, 1)))
    # visible positions of each (sequence, query row), padded with -1
    lists = []
    for b in range(B):
        L = int(lens[b])
        for i in range(n_q):
            last = L - n_q + i if causal else L - 1
            lists.append(np.nonzero(on_pool[b, :max(0, min(L, last + 1))])[0])
    K = max(1, max(len(c) for c in lists))
    idx = np.full((B * n_q, K), -1, dtype=np.int32)
    for r, cells in enumerate(lists):
        idx[r, :len(cells)] = cells
    return gather(qa, k_log, v_log, idx.reshape(B, n_q, K), scale, ks_log, vs_log,
                  _lib_override=_lib_override)


def gather(q, k, v, idx, scale, k_scale=None, v_scale=None, bias=None,
           _lib_override=None):
    """fp64 attention over the cache rows named by ``idx`` [B, n_q, K].

    One list per (sequence, query row), shared by every head of that row;
    entries < 0 or >= cap are skipped.  ``bias`` (optional, fp32 [B, n_q, K])
    is added to the score of each list entry ("qwen4exp : gather-based sparse
    attention for QSA decode", llama.cpp #28213, Overview: the mask entries
    travel with the gathered cells); an entry whose bias is -inf is dropped.
    Returns float64 [B, n_q, Hq, d].
    """
    lib = _lib_override or _load()
    qa = _as_np(q)
    if qa.dtype != np.uint16:
        raise TypeError("q must be bf16")
    ka, va, ksa, vsa, int8 = _kv_args(k, v, k_scale, v_scale)
    B, n_q, Hq, d = qa.shape
    _, Hkv, cap, d2 = ka.shape
    if d2 != d or va.shape != ka.shape:
        raise ValueError("shape mismatch")
    ia = np.ascontiguousarray(np.asarray(_as_np(idx), dtype=np.int32))
    if ia.ndim != 3 or ia.shape[:2] != (B, n_q):
        raise ValueError("idx must be [B, n_q, K]")
    K = ia.shape[2]
    out = np.zeros((B, n_q, Hq, d), dtype=np.float64)
    qs, ks, vs = _strides(qa), _strides(ka), _strides(va)
    ss = _strides(ksa) if int8 else np.zeros(3, dtype=np.int64)
    if bias is None:
        rc = lib.fdo_gather(_ptr(qa), _ptr(qs), _ptr(ka), _ptr(ks), _ptr(va),
                            _ptr(vs), int8,
                            _ptr(ksa) if int8 else None,
                            _ptr(vsa) if int8 else None, _ptr(ss), _ptr(ia), K,
                            B, n_q, Hq, Hkv, d, cap, float(scale), _ptr(out))
    else:
        ba = np.ascontiguousarray(np.asarray(_as_np(bias), dtype=np.float32))
        if ba.shape != ia.shape:
            raise ValueError("bias must be [B, n_q, K] like idx")
        rc = lib.fdo_gather_bias(_ptr(qa), _ptr(qs), _ptr(ka), _ptr(ks), _ptr(va),
                                 _ptr(vs), int8,
                                 _ptr(ksa) if int8 else None,
                                 _ptr(vsa) if int8 else None, _ptr(ss), _ptr(ia),
                                 _ptr(ba), K, B, n_q, Hq, Hkv, d, cap, float(scale),
                                 _ptr(out))
    if rc != 0:
        raise RuntimeError("fdo_gather failed: %d" % rc)
    return out
