"""Pins for the paged-cache oracle (no GPU).

``oracle.paged`` assembles each sequence's logical cache through the block
table and hands the visible positions to ``oracle.gather``.  These tests tie
it to things it does not compute itself: torch SDPA in float64 over a flat
cache whose pages were cut out with ``reshape`` and scattered by a seeded
permutation (so a wrong page index, row index or transposed table fails),
masks built by hand for bad table entries, and the invariants of the paged
layout (page order, poisoned free rows, rollback, clamping).
"""
import numpy as np
import pytest
import torch

import oracle
from decode_attention_preallocated_gb300 import workloads as W
from test_oracle_pins import TIGHT, dense_mask, dq, sdpa_masked


def to_pages(x, ps, perm):
    """Flat cache [B, H, cap, ...] -> (pool [B*cap/ps, H, ps, ...], table
    [B, cap/ps]): page i of sequence b is cut out by a reshape and stored at
    pool slot perm[b * (cap/ps) + i]."""
    B, H, cap = x.shape[:3]
    mp = cap // ps
    rest = tuple(x.shape[3:])
    pages = x.reshape(B, H, mp, ps, *rest).transpose(1, 2).reshape(B * mp, H, ps, *rest)
    pool = torch.empty_like(pages)
    pool[perm] = pages
    return pool, perm.view(B, mp).to(torch.int32)


def paged_from_flat(inp, ps, seed):
    B, cap = inp.k.shape[0], inp.k.shape[2]
    perm = torch.randperm(B * (cap // ps), generator=torch.Generator().manual_seed(seed))
    kp, table = to_pages(inp.k.contiguous(), ps, perm)
    vp, _ = to_pages(inp.v.contiguous(), ps, perm)
    ksp = vsp = None
    if inp.k_scale is not None:
        ksp, _ = to_pages(inp.k_scale.contiguous(), ps, perm)
        vsp, _ = to_pages(inp.v_scale.contiguous(), ps, perm)
    return kp, vp, ksp, vsp, table


def run_paged(inp, kp, vp, table, ksp=None, vsp=None, lengths=None):
    lens = inp.kv_lengths if lengths is None else torch.tensor(lengths, dtype=torch.int32)
    return torch.from_numpy(oracle.paged(inp.q, kp, vp, table, lens, inp.n_q, inp.causal,
                                         inp.scale, ksp, vsp))


@pytest.mark.parametrize("ps", [1, 3, 4, 12, 24])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("int8", [False, True])
def test_paged_matches_sdpa_on_the_flat_cache(ps, causal, int8):
    cap, lengths = 24, (19, 24, 5)
    inp = W.dense_inputs(3, 3, 6, 2, 16, cap, list(lengths), 40 + ps, causal, int8=int8)
    kp, vp, ksp, vsp, table = paged_from_flat(inp, ps, 7 + ps)
    out = run_paged(inp, kp, vp, table, ksp, vsp)
    ref = sdpa_masked(inp.q.double(), dq(inp.k, inp.k_scale), dq(inp.v, inp.v_scale),
                      dense_mask(lengths, 3, cap, causal), inp.scale)
    torch.testing.assert_close(out, ref, rtol=0, atol=TIGHT)


def test_token_major_pool_matches_head_major():
    inp = W.paged_inputs(2, 2, 8, 2, 16, 5, 6, [29, 11], 3, True)
    ref = run_paged(inp, inp.k, inp.v, inp.block_table)
    km = inp.k.transpose(1, 2).contiguous().transpose(1, 2)   # [P, ps, Hkv, d] storage
    vm = inp.v.transpose(1, 2).contiguous().transpose(1, 2)
    assert km.stride(2) == 2 * 16
    got = run_paged(inp, km, vm, inp.block_table)
    torch.testing.assert_close(got, ref, rtol=0, atol=0)


def test_bad_table_entry_skips_its_positions():
    cap, ps, lengths = 24, 4, (22, 17)
    inp = W.dense_inputs(2, 2, 4, 2, 8, cap, list(lengths), 51, True)
    kp, vp, _, _, table = paged_from_flat(inp, ps, 52)
    table = table.clone()
    table[0, 2] = -1                   # positions 8..11 of sequence 0
    table[1, 1] = kp.shape[0] + 5      # positions 4..7 of sequence 1
    table[1, 5] = -7                   # past the length: never consulted
    out = run_paged(inp, kp, vp, table)
    mask = dense_mask(lengths, 2, cap, True)
    mask[0, :, 8:12] = False
    mask[1, :, 4:8] = False
    ref = sdpa_masked(inp.q.double(), inp.k.double(), inp.v.double(), mask, inp.scale)
    torch.testing.assert_close(out, ref, rtol=0, atol=TIGHT)


def test_every_visible_page_bad_gives_zeros():
    inp = W.paged_inputs(1, 2, 4, 1, 8, 4, 3, [10], 5, False)
    table = torch.full_like(inp.block_table, -1)
    out = run_paged(inp, inp.k, inp.v, table)
    assert torch.count_nonzero(out) == 0


@pytest.mark.parametrize("int8", [False, True])
def test_free_rows_and_spare_pages_do_not_matter(int8):
    clean = W.paged_inputs(2, 3, 6, 2, 16, 7, 5, [30, 8], 61, True, int8=int8)
    poisoned = W.paged_inputs(2, 3, 6, 2, 16, 7, 5, [30, 8], 61, True, int8=int8, tail="nan")
    a = run_paged(clean, clean.k, clean.v, clean.block_table, clean.k_scale, clean.v_scale)
    b = run_paged(poisoned, poisoned.k, poisoned.v, poisoned.block_table,
                  poisoned.k_scale, poisoned.v_scale)
    assert torch.isfinite(b).all()
    torch.testing.assert_close(b, a, rtol=0, atol=0)


def test_page_order_in_the_pool_does_not_matter():
    inp = W.paged_inputs(2, 2, 4, 2, 8, 3, 6, [17, 12], 71, True)
    ref = run_paged(inp, inp.k, inp.v, inp.block_table)
    P = inp.k.shape[0]
    sigma = torch.randperm(P, generator=torch.Generator().manual_seed(72))
    k2 = torch.empty_like(inp.k)
    v2 = torch.empty_like(inp.v)
    k2[sigma] = inp.k
    v2[sigma] = inp.v
    table2 = sigma[inp.block_table.long()].to(torch.int32)
    got = run_paged(inp, k2, v2, table2)
    torch.testing.assert_close(got, ref, rtol=0, atol=0)


def test_rollback_and_clamping():
    cap, ps = 24, 6
    inp = W.dense_inputs(2, 2, 4, 2, 8, cap, [20, 24], 81, True)
    kp, vp, _, _, table = paged_from_flat(inp, ps, 82)
    # rollback: a shorter length sees exactly the shorter prefix
    short = run_paged(inp, kp, vp, table, lengths=[13, 7])
    ref = sdpa_masked(inp.q.double(), inp.k.double(), inp.v.double(),
                      dense_mask((13, 7), 2, cap, True), inp.scale)
    torch.testing.assert_close(short, ref, rtol=0, atol=TIGHT)
    # lengths past max_pages * page_size are clamped
    over = run_paged(inp, kp, vp, table, lengths=[cap + 9, -3])
    ref = sdpa_masked(inp.q.double(), inp.k.double(), inp.v.double(),
                      dense_mask((cap, 0), 2, cap, True), inp.scale)
    torch.testing.assert_close(over, ref, rtol=0, atol=TIGHT)


def test_paged_recipe_shapes():
    inp = W.paged_inputs(3, 2, 8, 2, 128, 64, 4, [100, 256, 1], 9, True, spare_pages=5)
    assert inp.k.shape == (3 * 4 + 5, 2, 64, 128)
    assert inp.block_table.shape == (3, 4)
    t = inp.block_table.flatten().tolist()
    assert len(set(t)) == len(t) and min(t) >= 0 and max(t) < inp.k.shape[0]
    assert inp.shape["cap"] == 256


def test_int8_token_major_pool_matches_head_major():
    inp = W.paged_inputs(2, 3, 8, 2, 16, 7, 6, [40, 9], 91, True, int8=True)
    ref = run_paged(inp, inp.k, inp.v, inp.block_table, inp.k_scale, inp.v_scale)
    km = inp.k.transpose(1, 2).contiguous().transpose(1, 2)
    vm = inp.v.transpose(1, 2).contiguous().transpose(1, 2)
    ksm = inp.k_scale.transpose(1, 2).contiguous().transpose(1, 2)
    vsm = inp.v_scale.transpose(1, 2).contiguous().transpose(1, 2)
    got = run_paged(inp, km, vm, inp.block_table, ksm, vsm)
    torch.testing.assert_close(got, ref, rtol=0, atol=0)


def test_poisoned_recipe_touches_only_free_rows():
    lens = [45, 3]
    inp = W.paged_inputs(2, 1, 4, 2, 8, 8, 6, lens, 92, False, tail="nan")
    P, Hkv, ps, d = inp.k.shape
    used = torch.zeros(P, ps, dtype=torch.bool)
    for b, L in enumerate(lens):
        for j in range(L):
            used[int(inp.block_table[b, j // ps]), j % ps] = True
    nan_rows = torch.isnan(inp.k).all(dim=-1).all(dim=1)     # [P, ps]
    assert torch.equal(nan_rows, ~used)
    assert torch.isfinite(inp.k[used.unsqueeze(1).expand(P, Hkv, ps)]).all()
