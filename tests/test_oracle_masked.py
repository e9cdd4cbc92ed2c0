"""Pins for the masked-prefix oracle (no GPU): torch SDPA in float64 with
the mask added to a hand-built window mask, a zero mask giving the dense
result bit for bit, -inf entries giving the dense result with those
positions removed, and a mask hiding everything giving zeros."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from decode_attention_preallocated_gb300 import workloads as W
from test_oracle_pins import TIGHT, dense_mask, sdpa_masked


def sdpa_additive(inp, mask, causal):
    """SDPA in float64 with (window mask) + (additive mask); rows with
    nothing visible -> 0."""
    B, n_q, Hq, d = inp.q.shape
    cap = inp.k.shape[2]
    win = dense_mask([int(x) for x in inp.kv_lengths], n_q, cap, causal)
    m = mask.double().clone()
    visible = win & torch.isfinite(m)
    m = torch.where(visible, m, torch.full_like(m, -1e300))
    g = Hq // inp.k.shape[1]
    kk = inp.k.double().repeat_interleave(g, dim=1)
    vv = inp.v.double().repeat_interleave(g, dim=1)
    out = F.scaled_dot_product_attention(inp.q.double().permute(0, 2, 1, 3), kk, vv,
                                         attn_mask=m[:, None].expand(B, Hq, n_q, cap),
                                         scale=inp.scale).permute(0, 2, 1, 3).contiguous()
    out[(~visible.any(dim=-1))[:, :, None, None].expand_as(out)] = 0.0
    return out


@pytest.mark.parametrize("causal,n_q", [(False, 1), (True, 3), (True, 6)])
def test_masked_matches_sdpa_with_an_additive_mask(causal, n_q):
    cap = 96
    inp = W.dense_inputs(3, n_q, 6, 2, 16, cap, [90, 0, 41], 110 + n_q, causal)
    g = torch.Generator().manual_seed(111)
    mask = torch.randn(3, n_q, cap, generator=g) * 2.0
    mask[torch.rand(3, n_q, cap, generator=g) < 0.5] = -float("inf")
    mask[0, :, 32:64] = -float("inf")                 # a whole chunk hidden
    out = oracle.masked(inp.q, inp.k, inp.v, inp.kv_lengths, mask, n_q, causal, inp.scale)
    torch.testing.assert_close(torch.from_numpy(out), sdpa_additive(inp, mask, causal),
                               rtol=0, atol=TIGHT)


def test_zero_mask_is_the_dense_result():
    inp = W.dense_inputs(2, 4, 8, 2, 16, 70, [70, 33], 112, True)
    mask = torch.zeros(2, 4, 70)
    got = oracle.masked(inp.q, inp.k, inp.v, inp.kv_lengths, mask, 4, True, inp.scale)
    ref = oracle.dense(inp.q, inp.k, inp.v, inp.kv_lengths, 4, True, inp.scale)
    np.testing.assert_array_equal(got, ref)


def test_neg_inf_removes_positions_and_everything_hidden_gives_zeros():
    cap = 50
    inp = W.dense_inputs(1, 2, 4, 1, 8, cap, [50], 113, False)
    mask = torch.zeros(1, 2, cap)
    mask[0, 0, 10:20] = -float("inf")
    mask[0, 1, :] = -float("inf")
    got = oracle.masked(inp.q, inp.k, inp.v, inp.kv_lengths, mask, 2, False, inp.scale)
    vis = dense_mask([50], 2, cap, False)
    vis[0, 0, 10:20] = False
    vis[0, 1, :] = False
    ref = sdpa_masked(inp.q.double(), inp.k.double(), inp.v.double(), vis, inp.scale)
    torch.testing.assert_close(torch.from_numpy(got), ref, rtol=0, atol=TIGHT)
    assert np.count_nonzero(got[0, 1]) == 0
