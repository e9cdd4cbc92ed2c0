"""Pins for the fused-append oracle (no GPU).

``oracle.append`` writes the new rows into a copy of the cache with a loop
and calls ``oracle.dense``.  These tests tie it to other constructions:
torch SDPA in float64 over keys built by concatenating the old prefix and
the new rows, the cache state after the step checked row by row against the
inputs, and sequential decoding (two one-row steps equal one two-row causal
step, row by row).
"""
import numpy as np
import pytest
import torch

import oracle
from decode_attention_preallocated_gb300 import workloads as W
from test_oracle_pins import TIGHT, sdpa_masked


def new_rows(B, n, Hkv, d, seed):
    g = torch.Generator().manual_seed(seed)
    return W.randn_bf16((B, n, Hkv, d), g, "cpu"), W.randn_bf16((B, n, Hkv, d), g, "cpu")


def concat_reference(inp, kn, vn, causal):
    """SDPA over [old prefix ; new rows] per sequence, padded to one length."""
    B, n, Hq, d = inp.q.shape
    lens = [int(x) for x in inp.kv_lengths]
    Lmax = max(lens) + n
    Hkv = inp.k.shape[1]
    K = torch.zeros(B, Hkv, Lmax, d, dtype=torch.float64)
    V = torch.zeros_like(K)
    mask = torch.zeros(B, n, Lmax, dtype=torch.bool)
    for b, L in enumerate(lens):
        kk = torch.cat([inp.k[b, :, :L].double(), kn[b].transpose(0, 1).double()], dim=1)
        vv = torch.cat([inp.v[b, :, :L].double(), vn[b].transpose(0, 1).double()], dim=1)
        K[b, :, : L + n] = kk
        V[b, :, : L + n] = vv
        for i in range(n):
            mask[b, i, : (L + i + 1 if causal else L + n)] = True
    return sdpa_masked(inp.q.double(), K, V, mask, inp.scale)


@pytest.mark.parametrize("n,causal", [(1, False), (1, True), (3, True), (6, True), (4, False)])
def test_append_matches_sdpa_over_concatenation(n, causal):
    cap = 40
    inp = W.dense_inputs(3, n, 6, 2, 16, cap, [17, 0, 33], 90 + n, causal)
    kn, vn = new_rows(3, n, 2, 16, 91)
    out, _, _, after = oracle.append(inp.q, inp.k, inp.v, kn, vn, inp.kv_lengths, causal,
                                     inp.scale)
    assert after.tolist() == [17 + n, n, 33 + n]
    ref = concat_reference(inp, kn, vn, causal)
    torch.testing.assert_close(torch.from_numpy(out), ref, rtol=0, atol=TIGHT)


def test_cache_after_the_step_holds_the_new_rows_and_nothing_else_changes():
    inp = W.dense_inputs(2, 4, 8, 2, 8, 30, [5, 21], 93, True)
    kn, vn = new_rows(2, 4, 2, 8, 94)
    _, ka, va, _ = oracle.append(inp.q, inp.k, inp.v, kn, vn, inp.kv_lengths, True, inp.scale)
    k0 = inp.k.view(torch.int16).numpy().view(np.uint16)
    v0 = inp.v.view(torch.int16).numpy().view(np.uint16)
    knb = kn.view(torch.int16).numpy().view(np.uint16)
    vnb = vn.view(torch.int16).numpy().view(np.uint16)
    for b, L in enumerate([5, 21]):
        for pos in range(30):
            if L <= pos < L + 4:
                assert np.array_equal(ka[b, :, pos], knb[b, pos - L])
                assert np.array_equal(va[b, :, pos], vnb[b, pos - L])
            else:
                assert np.array_equal(ka[b, :, pos], k0[b, :, pos])
                assert np.array_equal(va[b, :, pos], v0[b, :, pos])


def test_two_one_row_steps_equal_one_two_row_causal_step():
    inp = W.dense_inputs(2, 2, 8, 2, 16, 50, [12, 30], 95, True)
    kn, vn = new_rows(2, 2, 2, 16, 96)
    both, kb, vb, after = oracle.append(inp.q, inp.k, inp.v, kn, vn, inp.kv_lengths, True,
                                        inp.scale)
    o1, k1, v1, l1 = oracle.append(inp.q[:, :1], inp.k, inp.v, kn[:, :1], vn[:, :1],
                                   inp.kv_lengths, True, inp.scale)
    k1t = torch.from_numpy(k1.view(np.int16)).view(torch.bfloat16)
    v1t = torch.from_numpy(v1.view(np.int16)).view(torch.bfloat16)
    o2, k2, v2, l2 = oracle.append(inp.q[:, 1:], k1t, v1t, kn[:, 1:], vn[:, 1:], l1, True,
                                   inp.scale)
    assert np.array_equal(kb, k2) and np.array_equal(vb, v2)
    assert after.tolist() == l2.tolist()
    np.testing.assert_allclose(both[:, :1], o1, rtol=0, atol=TIGHT)
    np.testing.assert_allclose(both[:, 1:], o2, rtol=0, atol=TIGHT)


def test_rows_past_the_capacity_are_dropped_and_the_length_clamped():
    cap = 20
    inp = W.dense_inputs(1, 4, 4, 1, 8, cap, [18], 97, True)
    kn, vn = new_rows(1, 4, 1, 8, 98)
    out, ka, _, after = oracle.append(inp.q, inp.k, inp.v, kn, vn, inp.kv_lengths, True,
                                      inp.scale)
    assert after.tolist() == [cap]
    knb = kn.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ka[0, :, 18], knb[0, 0]) and np.array_equal(ka[0, :, 19], knb[0, 1])
    # the same as a dense call over the first cap positions of the written cache
    kat = torch.from_numpy(ka.view(np.int16)).view(torch.bfloat16)
    _, _, va, _ = oracle.append(inp.q, inp.k, inp.v, kn, vn, inp.kv_lengths, True, inp.scale)
    vat = torch.from_numpy(va.view(np.int16)).view(torch.bfloat16)
    ref = oracle.dense(inp.q, kat, vat, torch.tensor([cap], dtype=torch.int32), 4, True,
                       inp.scale)
    np.testing.assert_array_equal(out, ref)
