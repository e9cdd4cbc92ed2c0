"""The C ABI without a GPU: the library builds and loads, exports every
symbol include/fd.h declares, rejects bad arguments on the host before any
CUDA call, and its host partitioner mirror covers every tile exactly once."""
import ctypes
import os
import random
import re

import pytest

from decode_attention_preallocated_gb300 import build as fdbuild
from decode_attention_preallocated_gb300 import fd

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "fd.h")


@pytest.fixture(scope="module")
def L():
    fdbuild.build()
    return fd.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fd_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported_and_bound(L):
    names = declared_functions()
    assert "fd_decode" in names and "fd_decode_gather" in names
    bound = {n for n, _, _ in fd._SIGNATURES}
    for n in names:
        assert hasattr(L, n), "libfd.so does not export " + n
        assert n in bound, "binding does not declare " + n


def test_version_and_status_strings(L):
    assert L.fd_version() >= 1
    for code in (0, -1, -2, -3, -4, -5):
        assert fd.status_string(code) not in ("", "unknown status")
    assert fd.status_string(-99) == "unknown status"


def fake(shape, dtype=fd.FD_BF16, strides=None, ptr=0x100000):
    t = fd.FdTensor()
    t.data = ptr
    t.dtype = dtype
    t.ndim = len(shape)
    if strides is None:
        strides, acc = [], 1
        for s in reversed(shape):
            strides.insert(0, acc)
            acc *= s
    for i, (s, st) in enumerate(zip(shape, strides)):
        t.shape[i], t.stride[i] = s, st
    return t


def call_dense(q, k, v, out, n_q=1, causal=0, ws=None, lens=0x200000, opts=True, **kw):
    o = fd.FdOpts()
    o.ws = ws
    for key, val in kw.items():
        setattr(o, key, val)
    return fd.lib().fd_decode(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), lens,
                              n_q, causal, 0.1, ctypes.byref(out),
                              ctypes.byref(o) if opts else None)


def good(B=1, n_q=1, Hq=8, Hkv=2, d=128, cap=64):
    return (fake([B, n_q, Hq, d]), fake([B, Hkv, cap, d]), fake([B, Hkv, cap, d]),
            fake([B, n_q, Hq, d]))


def test_host_validation_codes(L):
    q, k, v, o = good()
    # all arguments valid but no workspace: rejected before any CUDA call
    assert call_dense(q, k, v, o) == fd.FD_ERR_WORKSPACE
    assert call_dense(q, k, v, o, opts=False) == fd.FD_ERR_ARG
    assert call_dense(q, k, v, o, lens=None) == fd.FD_ERR_ARG
    assert call_dense(q, k, v, o, n_q=2) == fd.FD_ERR_ARG          # n_q != q.shape[1]
    assert call_dense(q, k, v, o, causal=3) == fd.FD_ERR_ARG
    assert call_dense(q, k, v, o, kernel=7) == fd.FD_ERR_ARG
    assert call_dense(q, k, v, o, num_ctas=-1) == fd.FD_ERR_ARG
    assert call_dense(q, k, v, o, wait_limit_us=-1) == fd.FD_ERR_ARG
    assert call_dense(q, k, v, o, wait_limit_us=2000001) == fd.FD_ERR_ARG
    assert call_dense(q, k, v, o, wait_limit_us=1000) == fd.FD_ERR_WORKSPACE
    o2 = fd.FdOpts()
    o2.reserved[1] = 1
    assert fd.lib().fd_decode(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), 0x200000, 1, 0,
                              0.1, ctypes.byref(o), ctypes.byref(o2)) == fd.FD_ERR_ARG
    assert L.fd_workspace_fill_counters(None, -1, None) == fd.FD_ERR_ARG
    qq, kk, vv, oo = good(d=64)
    assert call_dense(qq, kk, vv, oo) == fd.FD_ERR_UNSUPPORTED
    qq, kk, vv, oo = good(n_q=7)
    assert call_dense(qq, kk, vv, oo, n_q=7) == fd.FD_ERR_UNSUPPORTED
    qq, kk, vv, oo = good(Hq=6, Hkv=4)
    assert call_dense(qq, kk, vv, oo) == fd.FD_ERR_ARG              # Hq % Hkv
    qq, kk, vv, oo = good(Hq=72, Hkv=1)
    assert call_dense(qq, kk, vv, oo) == fd.FD_ERR_UNSUPPORTED      # 72 rows > 64
    # misaligned cache pointer / stride
    q, k, v, o = good()
    k.data = 0x100008
    assert call_dense(q, k, v, o) == fd.FD_ERR_ALIGN
    q, k, v, o = good()
    k2 = fake([1, 2, 64, 128], strides=[2 * 64 * 132, 64 * 132, 132, 1])
    assert call_dense(q, k2, k2, o) == fd.FD_ERR_ALIGN
    # wrong dtypes / shapes / inner stride
    q, k, v, o = good()
    assert call_dense(q, fake([1, 2, 64, 128], fd.FD_F32), v, o) == fd.FD_ERR_ARG
    assert call_dense(q, k, v, fake([1, 1, 8, 128], fd.FD_I8)) == fd.FD_ERR_ARG
    assert call_dense(q, k, fake([1, 2, 32, 128]), o) == fd.FD_ERR_ARG
    assert call_dense(q, k, v, fake([1, 1, 8, 128], strides=[1024, 1024, 128, 2])) == fd.FD_ERR_ARG
    q, k, v, o = good()
    q.data = None
    assert call_dense(q, k, v, o) == fd.FD_ERR_ARG


def test_int8_and_gather_validation(L):
    q, _, _, o = good()
    k8 = fake([1, 2, 64, 128], fd.FD_I8)
    ks = fake([1, 2, 64], fd.FD_F32)
    op = fd.FdOpts()
    rc = L.fd_decode_int8(ctypes.byref(q), ctypes.byref(k8), ctypes.byref(k8),
                          ctypes.byref(ks), ctypes.byref(ks), 0x200000, 1, 0, 0.1,
                          ctypes.byref(o), ctypes.byref(op))
    assert rc == fd.FD_ERR_WORKSPACE
    bad = fake([1, 2, 63], fd.FD_F32)
    rc = L.fd_decode_int8(ctypes.byref(q), ctypes.byref(k8), ctypes.byref(k8),
                          ctypes.byref(bad), ctypes.byref(ks), 0x200000, 1, 0, 0.1,
                          ctypes.byref(o), ctypes.byref(op))
    assert rc == fd.FD_ERR_ARG
    _, k, v, _ = good()
    rc = L.fd_decode_gather(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), 0x300000,
                            16, ctypes.byref(o), ctypes.byref(op))
    assert rc == fd.FD_ERR_WORKSPACE
    rc = L.fd_decode_gather(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), None,
                            16, ctypes.byref(o), ctypes.byref(op))
    assert rc == fd.FD_ERR_ARG


def call_paged(q, k, v, out, table=0x400000, max_pages=4, ks=None, vs=None, n_q=1,
               causal=0, lens=0x200000):
    op = fd.FdOpts()
    return fd.lib().fd_decode_paged(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v),
                                    ctypes.byref(ks) if ks is not None else None,
                                    ctypes.byref(vs) if vs is not None else None,
                                    table, max_pages, lens, n_q, causal, 0.1,
                                    ctypes.byref(out), ctypes.byref(op))


def test_paged_validation(L):
    # pools [num_pages, Hkv, page_size, d]; the batch comes from q
    q, _, _, o = fake([3, 1, 8, 128]), None, None, fake([3, 1, 8, 128])
    kp = fake([10, 2, 16, 128])
    assert call_paged(q, kp, kp, o) == fd.FD_ERR_WORKSPACE        # valid up to the workspace
    assert call_paged(q, kp, kp, o, table=None) == fd.FD_ERR_ARG
    assert call_paged(q, kp, kp, o, max_pages=0) == fd.FD_ERR_ARG
    assert call_paged(q, kp, kp, o, lens=None) == fd.FD_ERR_ARG
    assert call_paged(q, kp, kp, o, causal=2) == fd.FD_ERR_ARG
    assert call_paged(q, kp, fake([10, 2, 8, 128]), o) == fd.FD_ERR_ARG   # k / v pools differ
    assert call_paged(q, fake([0, 2, 16, 128]), fake([0, 2, 16, 128]), o) == fd.FD_ERR_ARG
    assert call_paged(q, kp, kp, o, max_pages=(1 << 31) // 16) == fd.FD_ERR_UNSUPPORTED
    ks = fake([10, 2, 16], fd.FD_F32)
    assert call_paged(q, kp, kp, o, ks=ks, vs=ks) == fd.FD_ERR_ARG    # scales on a bf16 pool
    k8 = fake([10, 2, 16, 128], fd.FD_I8)
    assert call_paged(q, k8, k8, o, ks=ks, vs=ks) == fd.FD_ERR_WORKSPACE
    assert call_paged(q, k8, k8, o) == fd.FD_ERR_ARG                  # int8 pool, no scales
    bad = fake([10, 2, 15], fd.FD_F32)
    assert call_paged(q, k8, k8, o, ks=bad, vs=ks) == fd.FD_ERR_ARG
    k2 = fake([10, 2, 16, 128], strides=[2 * 16 * 132, 16 * 132, 132, 1])
    assert call_paged(q, k2, k2, o) == fd.FD_ERR_ALIGN


def test_append_validation(L):
    q, k, v, o = good(B=2, n_q=3)
    kn = fake([2, 3, 2, 128])
    op = fd.FdOpts()

    def call(kn_, vn_, update=1, lens=0x200000, causal=1):
        return L.fd_decode_append(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v),
                                  ctypes.byref(kn_), ctypes.byref(vn_), lens, update, causal,
                                  0.1, ctypes.byref(o), ctypes.byref(op))

    q, k, v, o = good(B=2, n_q=3)
    assert call(kn, kn) == fd.FD_ERR_WORKSPACE                  # valid up to the workspace
    assert call(kn, kn, update=2) == fd.FD_ERR_ARG
    assert call(kn, kn, lens=None) == fd.FD_ERR_ARG
    assert call(fake([2, 2, 2, 128]), kn) == fd.FD_ERR_ARG       # n_new != n_q
    assert call(kn, fake([2, 3, 1, 128])) == fd.FD_ERR_ARG       # Hkv
    assert call(fake([2, 3, 2, 128], fd.FD_F32), kn) == fd.FD_ERR_ARG
    assert call(fake([2, 3, 2, 128], ptr=0x100008), kn) == fd.FD_ERR_ALIGN
    assert call(fake([2, 3, 2, 128], strides=[3 * 2 * 132, 2 * 132, 132, 1]), kn) == fd.FD_ERR_ALIGN
    k8 = fake([2, 2, 64, 128], fd.FD_I8)
    rc = L.fd_decode_append(ctypes.byref(q), ctypes.byref(k8), ctypes.byref(k8),
                            ctypes.byref(kn), ctypes.byref(kn), 0x200000, 1, 1, 0.1,
                            ctypes.byref(o), ctypes.byref(op))
    assert rc == fd.FD_ERR_ARG                                   # bf16 caches only


def test_masked_validation(L):
    q, k, v, o = good(B=2, n_q=3, cap=64)
    m = fake([2, 3, 64], fd.FD_F32)
    op = fd.FdOpts()

    def call(mask, lens=0x200000, k_=k):
        return L.fd_decode_masked(ctypes.byref(q), ctypes.byref(k_), ctypes.byref(k_), lens,
                                  ctypes.byref(mask) if mask is not None else None, 3, 1, 0.1,
                                  ctypes.byref(o), ctypes.byref(op))

    assert call(m) == fd.FD_ERR_WORKSPACE                         # valid up to the workspace
    assert call(None) == fd.FD_ERR_ARG
    assert call(m, lens=None) == fd.FD_ERR_ARG
    assert call(fake([2, 3, 63], fd.FD_F32)) == fd.FD_ERR_ARG      # not [B, n_q, cap]
    assert call(fake([2, 3, 64], fd.FD_BF16)) == fd.FD_ERR_ARG     # not fp32
    assert call(fake([2, 3, 64], fd.FD_F32, strides=[384, 128, 2])) == fd.FD_ERR_ARG
    assert call(fake([2, 3, 64], fd.FD_F32, ptr=0x100002)) == fd.FD_ERR_ALIGN
    assert call(m, k_=fake([2, 2, 64, 128], fd.FD_I8)) == fd.FD_ERR_ARG   # bf16 caches only


def test_topk_validation(L):
    # every check fails before anything is launched
    assert L.fd_topk_blocks(None, 1, 1, 8, 0x200000, 4, 2, 0x300000, None) == fd.FD_ERR_ARG
    assert L.fd_topk_blocks(0x100000, 1, 1, 8, None, 4, 2, 0x300000, None) == fd.FD_ERR_ARG
    assert L.fd_topk_blocks(0x100000, 1, 1, 8, 0x200000, 4, 2, None, None) == fd.FD_ERR_ARG
    assert L.fd_topk_blocks(0x100000, 0, 1, 8, 0x200000, 4, 2, 0x300000, None) == fd.FD_ERR_ARG
    assert L.fd_topk_blocks(0x100000, 1, 1, 8, 0x200000, 0, 2, 0x300000, None) == fd.FD_ERR_ARG
    assert L.fd_topk_blocks(0x100000, 1, 1, 8, 0x200000, 4, 0, 0x300000, None) == fd.FD_ERR_ARG
    assert L.fd_topk_blocks(0x100000, 1, 1, 32769, 0x200000, 4, 2, 0x300000,
                            None) == fd.FD_ERR_UNSUPPORTED
    assert L.fd_topk_blocks(0x100002, 1, 1, 8, 0x200000, 4, 2, 0x300000, None) == fd.FD_ERR_ALIGN


def test_workspace_size_formula(L):
    n = L.fd_workspace_bytes(10, 24, 256, 300)
    floats = (10 + 300) * 24 * 258
    assert n >= floats * 4 + 10 * 4 + 4
    assert n % 256 == 0
    assert L.fd_workspace_bytes(0, 1, 1, 1) == 0


def test_masked_list_size(L):
    # the list (ceil(cap / 32) entries per sequence, rounded up to 4), one
    # count per sequence, and the listing pass's staging area (256 entries and
    # one count per block of 256 chunks), all int32
    def expect(B, cap):
        nch = -(-cap // 32)
        nblk = -(-nch // 256)
        up4 = lambda x: -(-x // 4) * 4
        return 4 * (B * up4(nch) + up4(B) + B * nblk * 256 + up4(B * nblk))

    for B, cap in ((1, 131072), (8, 32768), (3, 20000), (1, 1), (5, 33), (65535, 4096),
                   (2, 1 << 23)):
        assert L.fd_masked_list_bytes(B, cap) == expect(B, cap), (B, cap)
        assert fd.masked_list_bytes(B, cap) == expect(B, cap)
    assert L.fd_masked_list_bytes(0, 64) == 0
    assert L.fd_masked_list_bytes(65536, 64) == 0
    assert L.fd_masked_list_bytes(1, 0) == 0
    assert L.fd_masked_list_bytes(1, (1 << 23) + 1) == 0    # more than 1024 listing blocks


@pytest.mark.parametrize("seed", range(40))
def test_partition_covers_each_tile_once(L, seed):
    rnd = random.Random(seed)
    nseg = rnd.randint(1, 40)
    tile = rnd.choice([16, 32, 64, 128])
    maxlen = 5000 if seed % 2 else 300           # odd seeds: more blocks than tiles
    lens = [rnd.choice([0, rnd.randint(1, maxlen)]) for _ in range(nseg)]
    grid = rnd.randint(1, 400)
    V = rnd.choice([0, 0, 1, 4, 6])      # units charged per segment start
    total, first, pieces = fd.plan(lens, tile, grid, V)
    ntiles = [-(-x // tile) for x in lens]
    units = [n + V if n else 0 for n in ntiles]
    assert total == sum(units)
    if total == 0:
        assert all(p == 0 for p in pieces)
        return
    G = min(grid, total)          # blocks beyond the unit count get no work
    starts = [c * total // G for c in range(G + 1)]
    assert all(starts[c + 1] > starts[c] for c in range(G))
    # balanced: block ranges differ by at most one unit
    sizes = [starts[c + 1] - starts[c] for c in range(G)]
    assert max(sizes) - min(sizes) <= 1
    seen = {}
    slots = set()
    u = 0                          # unit where segment s starts
    for s in range(nseg):
        if ntiles[s] == 0:
            assert pieces[s] == 0
            continue
        t0, t1 = u + V, u + units[s]     # units that carry the segment's tiles
        blocks = [c for c in range(G) if starts[c] < t1 and starts[c + 1] > t0]
        assert blocks == list(range(first[s], first[s] + pieces[s]))
        for c in blocks:
            lo, hi = max(starts[c], t0), min(starts[c + 1], t1)
            for x in range(lo - t0, hi - t0):
                seen[(s, x)] = seen.get((s, x), 0) + 1
            assert s + c not in slots          # workspace slot is unique
            slots.add(s + c)
            assert s + c < nseg + G - 1
        u += units[s]
    # every tile of every segment is covered exactly once
    assert len(seen) == sum(ntiles) and all(x == 1 for x in seen.values())
