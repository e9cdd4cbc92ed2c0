"""Seeded synthetic inputs for decode attention over a preallocated KV cache.

This module only makes inputs: shapes, seeded N(0,1) values, ragged length
mixes, top-k style index lists and the int8 cache writer.  It holds no
attention arithmetic, so both the CUDA path and any checker can draw the same
inputs from it.

Workload shapes (all values N(0,1) from ``torch.Generator.manual_seed``,
rounded to bf16 with round-to-nearest-even by ``Tensor.to``):

* ``dense_1k``   -- 1 sequence, 1 query row, 8 q heads / 2 kv heads,
  head_dim 128, capacity 4096 with 1000 filled, non-causal.
* ``mtp_verify`` -- 1 sequence, 4 query rows (token + 3 drafts,
  bottom-right causal), 16 / 4 heads, head_dim 256, capacity 24007, 3000
  filled.
* ``ragged``     -- 8 sequences, lengths uniform in [1024, 32768] from the
  seed, capacity 32768, 6-row causal window, 16 / 4 heads, head_dim 256.
* ``gather``     -- 1 sequence, 131072 cached tokens, 32 / 4 heads,
  head_dim 128, one list of 2048 distinct cells: the last 128 positions
  plus 1920 drawn uniformly without replacement from the rest, shuffled.
* ``int8``       -- 4 sequences x 131072 tokens, int8 K/V quantised per
  (token, kv head) with fp32 scales, 1 query row, 32 / 8 heads,
  head_dim 128.
* ``paged_ps<P>`` / ``paged_int8_ps<P>`` -- the ragged / int8 workloads over
  a paged cache: pools of P-position pages, every sequence's pages scattered
  over the pool by a seeded permutation (``paged_inputs``).

The ComfyUI issue's cache is "prompt + max_length + 7" long with only the
answer-so-far filled ("Qwen3.5 text generation attends over the full KV
capacity", problem statement); the unused tail here holds N(0,1) garbage or,
on request, NaN/Inf poison so any read of it that reaches the arithmetic
shows up in the output.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch


@dataclass
class DecodeInputs:
    q: torch.Tensor                 # [B, n_q, Hq, d] bf16
    k: torch.Tensor                 # [B, Hkv, cap, d] bf16 or int8 (maybe strided)
    v: torch.Tensor
    kv_lengths: torch.Tensor        # [B] int32 (same device as q)
    n_q: int
    causal: bool
    scale: float
    k_scale: Optional[torch.Tensor] = None   # [B, Hkv, cap] fp32 (int8 only)
    v_scale: Optional[torch.Tensor] = None
    idx: Optional[torch.Tensor] = None       # [B, n_q, K] int32 (gather only)
    lengths_host: list = field(default_factory=list)
    name: str = ""
    # paged caches: k, v (and the scales) are pools [num_pages, Hkv, page_size,
    # ...]; position j of sequence b is row j % page_size of page
    # block_table[b, j // page_size]
    block_table: Optional[torch.Tensor] = None   # [B, max_pages] int32
    page_size: int = 0
    # masked prefix: fp32 [B, n_q, cap] added to the scores (-inf hides)
    mask: Optional[torch.Tensor] = None

    @property
    def shape(self):
        B, n_q, Hq, d = self.q.shape
        cap = (self.block_table.shape[1] * self.page_size if self.block_table is not None
               else self.k.shape[2])
        return dict(B=B, n_q=n_q, Hq=Hq, Hkv=self.k.shape[1], d=d, cap=cap)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def randn_bf16(shape, gen, device, mult: float = 1.0) -> torch.Tensor:
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if mult != 1.0:
        x.mul_(mult)
    return x.to(torch.bfloat16)


def make_cache(B, Hkv, cap, d, gen, device, layout="bhtd", dtype=torch.bfloat16):
    """N(0,1) cache tensor viewed as [B, Hkv, cap, d].

    layout "bhtd": contiguous [B, Hkv, cap, d];
    layout "bthd": contiguous [B, cap, Hkv, d] seen through a transpose.
    """
    if layout == "bhtd":
        x = torch.randn((B, Hkv, cap, d), generator=gen, device=device)
        return x.to(dtype)
    if layout == "bthd":
        x = torch.randn((B, cap, Hkv, d), generator=gen, device=device)
        return x.to(dtype).transpose(1, 2)
    raise ValueError(layout)


def poison_tail(t: torch.Tensor, lengths, value=float("nan")) -> None:
    """Write ``value`` into every cache row at or past each sequence's length."""
    for b, L in enumerate(lengths):
        L = max(0, min(int(L), t.shape[2]))
        if L < t.shape[2]:
            t[b, :, L:, :] = value


def quantize_per_token(x: torch.Tensor):
    """Symmetric int8 cache writer, one scale per (token, kv head).

    scale = max_d |x| / 127; code = clamp(round_half_even(x / scale), -127, 127);
    an all-zero row gets scale 0 and zero codes.  This produces the int8
    cache's contents (the kernel only reads them); it is not timed.
    x: [B, Hkv, cap, d] float -> (int8 [B, Hkv, cap, d], fp32 [B, Hkv, cap]).
    """
    xf = x.float()
    amax = xf.abs().amax(dim=-1)
    scale = amax / 127.0
    safe = torch.where(scale > 0, scale, torch.ones_like(scale))
    codes = torch.round(xf / safe.unsqueeze(-1)).clamp_(-127, 127)
    codes = torch.where(scale.unsqueeze(-1) > 0, codes, torch.zeros_like(codes))
    return codes.to(torch.int8), scale.to(torch.float32)


def topk_like_indices(cap: int, K: int, recent: int, gen, n_lists: int = 1):
    """``n_lists`` lists of K distinct cells: the last ``recent`` positions
    plus K - recent drawn uniformly without replacement from [0, cap-recent),
    each list shuffled (int32 [n_lists, K], on the CPU)."""
    if K > cap or recent > K:
        raise ValueError("need recent <= K <= cap")
    out = torch.empty((n_lists, K), dtype=torch.int32)
    tail = torch.arange(cap - recent, cap, dtype=torch.int64)
    for n in range(n_lists):
        pick = torch.randperm(cap - recent, generator=gen)[: K - recent]
        cells = torch.cat([tail, pick])
        perm = torch.randperm(K, generator=gen)
        out[n] = cells[perm].to(torch.int32)
    return out


def dense_inputs(B, n_q, Hq, Hkv, d, cap, lengths, seed, causal,
                 device="cpu", layout="bhtd", tail="randn", q_mult=1.0,
                 scale=None, int8=False, name="") -> DecodeInputs:
    """Generic seeded dense-prefix (or int8) decode inputs."""
    gen = _gen(seed, "cpu" if str(device) == "cpu" else device)
    q = randn_bf16((B, n_q, Hq, d), gen, device, q_mult)
    if int8:
        src_k = make_cache(B, Hkv, cap, d, gen, device, layout, torch.float32)
        src_v = make_cache(B, Hkv, cap, d, gen, device, layout, torch.float32)
        k, ks = quantize_per_token(src_k)
        v, vs = quantize_per_token(src_v)
        if layout == "bthd":
            k = k.transpose(1, 2).contiguous().transpose(1, 2)
            v = v.transpose(1, 2).contiguous().transpose(1, 2)
        del src_k, src_v
    else:
        k = make_cache(B, Hkv, cap, d, gen, device, layout)
        v = make_cache(B, Hkv, cap, d, gen, device, layout)
        ks = vs = None
    lengths = [int(x) for x in lengths]
    if tail in ("nan", "inf"):
        if int8:
            # int8 codes cannot hold NaN; poison the scales instead
            poison_tail(ks.unsqueeze(-1), lengths, float(tail))
            poison_tail(vs.unsqueeze(-1), lengths, float(tail))
        else:
            poison_tail(k, lengths, float(tail))
            poison_tail(v, lengths, float("nan") if tail == "nan" else -float("inf"))
    lens = torch.tensor(lengths, dtype=torch.int32, device=device)
    return DecodeInputs(q=q, k=k, v=v, kv_lengths=lens, n_q=n_q,
                        causal=bool(causal),
                        scale=(1.0 / math.sqrt(d)) if scale is None else scale,
                        k_scale=ks, v_scale=vs, lengths_host=lengths, name=name)


def gather_inputs(B, n_q, Hq, Hkv, d, cap, K, recent, seed, device="cpu",
                  layout="bhtd", q_mult=1.0, name="", int8=False) -> DecodeInputs:
    """Seeded gather inputs: one top-k-like list of K distinct cells per
    (sequence, query row); int8=True quantises the caches per (token, kv
    head) as dense_inputs does."""
    gen = _gen(seed, "cpu" if str(device) == "cpu" else device)
    q = randn_bf16((B, n_q, Hq, d), gen, device, q_mult)
    ks = vs = None
    if int8:
        k, ks = quantize_per_token(make_cache(B, Hkv, cap, d, gen, device, layout, torch.float32))
        v, vs = quantize_per_token(make_cache(B, Hkv, cap, d, gen, device, layout, torch.float32))
        if layout == "bthd":
            k = k.transpose(1, 2).contiguous().transpose(1, 2)
            v = v.transpose(1, 2).contiguous().transpose(1, 2)
    else:
        k = make_cache(B, Hkv, cap, d, gen, device, layout)
        v = make_cache(B, Hkv, cap, d, gen, device, layout)
    cpu_gen = _gen(seed + 7919, "cpu")
    idx = topk_like_indices(cap, K, recent, cpu_gen, B * n_q).view(B, n_q, K)
    return DecodeInputs(q=q, k=k, v=v,
                        kv_lengths=torch.full((B,), cap, dtype=torch.int32, device=device),
                        n_q=n_q, causal=False, scale=1.0 / math.sqrt(d), k_scale=ks,
                        v_scale=vs, idx=idx.to(device), lengths_host=[cap] * B, name=name)


def paged_inputs(B, n_q, Hq, Hkv, d, page_size, max_pages, lengths, seed, causal,
                 device="cpu", layout="bhtd", spare_pages=3, tail="randn",
                 int8=False, name="") -> DecodeInputs:
    """Seeded decode inputs over a paged cache.

    Pools k, v: [num_pages, Hkv, page_size, d] with num_pages =
    B * max_pages + spare_pages (layout "bthd" stores [num_pages, page_size,
    Hkv, d] and returns the transposed view); int8 pools are written by
    ``quantize_per_token`` with fp32 scales [num_pages, Hkv, page_size].
    block_table [B, max_pages]: the first B * max_pages entries of a seeded
    permutation of the pool's pages, so a sequence's consecutive positions
    sit on scattered pages and the spare pages belong to no sequence.
    tail="nan"/"inf" poisons every pool row that holds no position below its
    sequence's length (the spare pages included).
    """
    gen = _gen(seed, "cpu" if str(device) == "cpu" else device)
    q = randn_bf16((B, n_q, Hq, d), gen, device)
    P = B * max_pages + spare_pages
    if int8:
        src_k = make_cache(P, Hkv, page_size, d, gen, device, layout, torch.float32)
        src_v = make_cache(P, Hkv, page_size, d, gen, device, layout, torch.float32)
        k, ks = quantize_per_token(src_k)
        v, vs = quantize_per_token(src_v)
        if layout == "bthd":
            k = k.transpose(1, 2).contiguous().transpose(1, 2)
            v = v.transpose(1, 2).contiguous().transpose(1, 2)
        del src_k, src_v
    else:
        k = make_cache(P, Hkv, page_size, d, gen, device, layout)
        v = make_cache(P, Hkv, page_size, d, gen, device, layout)
        ks = vs = None
    cpu_gen = _gen(seed + 104729, "cpu")
    table = torch.randperm(P, generator=cpu_gen)[: B * max_pages].view(B, max_pages)
    table = table.to(torch.int32)
    lengths = [int(x) for x in lengths]
    if tail in ("nan", "inf"):
        used = torch.zeros((P, page_size), dtype=torch.bool)
        for b, L in enumerate(lengths):
            for j in range(max(0, min(L, max_pages * page_size))):
                used[int(table[b, j // page_size]), j % page_size] = True
        free = (~used).to(k.device)
        if int8:
            # int8 codes cannot hold NaN; poison the scales instead
            ks[free.unsqueeze(1).expand_as(ks)] = float(tail)
            vs[free.unsqueeze(1).expand_as(vs)] = float(tail)
        else:
            m = free.unsqueeze(1).unsqueeze(-1).expand_as(k)
            k[m] = float(tail)
            v[m] = float("nan") if tail == "nan" else -float("inf")
    lens = torch.tensor(lengths, dtype=torch.int32, device=device)
    return DecodeInputs(q=q, k=k, v=v, kv_lengths=lens, n_q=n_q, causal=bool(causal),
                        scale=1.0 / math.sqrt(d), k_scale=ks, v_scale=vs,
                        lengths_host=lengths, name=name, block_table=table.to(device),
                        page_size=page_size)


def ragged_lengths(B, lo, hi, seed):
    g = _gen(seed, "cpu")
    return torch.randint(lo, hi + 1, (B,), generator=g).tolist()


# The five named workloads.  ``scale_down`` shrinks capacity/lengths for quick
# parity runs while keeping head counts, head_dim and window shape.
def workload(name: str, seed: int = 1, device="cpu", tail="randn",
             layout="bhtd") -> DecodeInputs:
    if name == "dense_1k":
        return dense_inputs(1, 1, 8, 2, 128, 4096, [1000], seed, False, device,
                            layout, tail, name=name)
    if name == "mtp_verify":
        return dense_inputs(1, 4, 16, 4, 256, 24007, [3000], seed, True, device,
                            layout, tail, name=name)
    if name.startswith("mtp_verify_cap"):
        # the MTP-verify workload in another capacity (the time and the bytes
        # read must not depend on it)
        cap = int(name[len("mtp_verify_cap"):])
        return dense_inputs(1, 4, 16, 4, 256, cap, [3000], seed, True, device,
                            layout, tail, name=name)
    if name == "ragged":
        lens = ragged_lengths(8, 1024, 32768, seed)
        return dense_inputs(8, 6, 16, 4, 256, 32768, lens, seed, True, device,
                            layout, tail, name=name)
    if name == "gather":
        return gather_inputs(1, 1, 32, 4, 128, 131072, 2048, 128, seed, device,
                             layout, name=name)
    if name == "int8":
        return dense_inputs(4, 1, 32, 8, 128, 131072, [131072] * 4, seed, False,
                            device, layout, tail, int8=True, name=name)
    if name == "int8_d256":
        # the int8 workload's shape at head_dim 256
        return dense_inputs(4, 1, 32, 8, 256, 131072, [131072] * 4, seed, False, device,
                            layout, tail, int8=True, name=name)
    if name == "gather_int8":
        # the gather workload over an int8 cache
        return gather_inputs(1, 1, 32, 4, 128, 131072, 2048, 128, seed, device, layout,
                             name=name, int8=True)
    if name == "masked_list":
        # the gather workload's selection as a mask over its whole prefix
        inp = gather_inputs(1, 1, 32, 4, 128, 131072, 2048, 128, seed, device, layout,
                            name=name)
        inp.mask = torch.full((1, 1, 131072), -float("inf"), device=device)
        inp.mask[0, 0, inp.idx[0, 0].long()] = 0.0
        inp.idx = None
        return inp
    if name.startswith("paged_ps"):
        # the ragged workload over a paged cache of page_size positions
        ps = int(name[len("paged_ps"):])
        lens = ragged_lengths(8, 1024, 32768, seed)
        return paged_inputs(8, 6, 16, 4, 256, ps, 32768 // ps, lens, seed, True, device,
                            layout, tail=tail, name=name)
    if name.startswith("paged_int8_ps"):
        # the int8 workload over a paged cache of page_size positions
        ps = int(name[len("paged_int8_ps"):])
        return paged_inputs(4, 1, 32, 8, 128, ps, 131072 // ps, [131072] * 4, seed, False,
                            device, layout, tail=tail, int8=True, name=name)
    raise KeyError(name)


WORKLOADS = ("dense_1k", "mtp_verify", "ragged", "gather", "int8")
# The ragged and int8 workloads over paged caches (page size 64 for bf16,
# 256 for int8; other page sizes by name, e.g. "paged_ps16").
PAGED_WORKLOADS = ("paged_ps64", "paged_int8_ps256")
