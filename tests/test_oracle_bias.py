"""Pins for the per-cell bias of the gather oracle (no GPU): torch SDPA in
float64 with an additive float mask, closed forms (zero and constant biases
change nothing; with identical keys, biases log w give the w-weighted mean of
the values) and the -inf rule (an entry with bias -inf is the same as no
entry)."""
import math

import numpy as np
import torch

import oracle
from decode_attention_preallocated_gb300 import workloads as W
from test_oracle_mutants import gather_bias_values
from test_oracle_pins import TIGHT, sdpa_bias


def test_biased_gather_matches_sdpa_with_an_additive_mask():
    inp = W.gather_inputs(2, 3, 8, 2, 16, 50, 14, 4, seed=31)
    bias = gather_bias_values(inp.idx, 32)
    out = oracle.gather(inp.q, inp.k, inp.v, inp.idx, inp.scale, bias=bias)
    ref = sdpa_bias(inp.q.double(), inp.k.double(), inp.v.double(), inp.idx, bias, 50,
                    inp.scale)
    torch.testing.assert_close(torch.from_numpy(out), ref, rtol=0, atol=TIGHT)
    assert np.count_nonzero(out[0, -1]) == 0          # every entry -inf: zeros


def test_zero_and_constant_biases_change_nothing():
    inp = W.gather_inputs(2, 2, 8, 2, 16, 40, 12, 4, seed=33)
    plain = oracle.gather(inp.q, inp.k, inp.v, inp.idx, inp.scale)
    zero = oracle.gather(inp.q, inp.k, inp.v, inp.idx, inp.scale,
                         bias=torch.zeros(inp.idx.shape))
    np.testing.assert_array_equal(zero, plain)
    const = oracle.gather(inp.q, inp.k, inp.v, inp.idx, inp.scale,
                          bias=torch.full(inp.idx.shape, 7.25))
    np.testing.assert_allclose(const, plain, rtol=0, atol=TIGHT)


def test_neg_inf_bias_equals_dropping_the_entry():
    inp = W.gather_inputs(1, 2, 4, 1, 8, 30, 10, 2, seed=35)
    bias = torch.zeros(inp.idx.shape)
    bias[0, 0, 2] = -float("inf")
    bias[0, 1, 7] = -float("inf")
    got = oracle.gather(inp.q, inp.k, inp.v, inp.idx, inp.scale, bias=bias)
    idx = inp.idx.clone()
    idx[0, 0, 2] = -1
    idx[0, 1, 7] = -1
    ref = oracle.gather(inp.q, inp.k, inp.v, idx, inp.scale)
    np.testing.assert_array_equal(got, ref)


def test_identical_keys_with_log_weights_give_the_weighted_mean():
    B, n_q, Hq, Hkv, d, cap = 1, 1, 2, 1, 8, 6
    g = torch.Generator().manual_seed(37)
    q = W.randn_bf16((B, n_q, Hq, d), g, "cpu")
    k = W.randn_bf16((1, 1, 1, d), g, "cpu").expand(B, Hkv, cap, d).contiguous()
    v = W.randn_bf16((B, Hkv, cap, d), g, "cpu")
    idx = torch.tensor([[[0, 2, 3, 5]]], dtype=torch.int32)
    w = [1.0, 2.0, 0.5, 4.0]
    bias = torch.tensor([[[math.log(x) for x in w]]], dtype=torch.float32)
    out = oracle.gather(q, k, v, idx, 0.3, bias=bias)
    wd = np.array([float(b) for b in bias[0, 0]], dtype=np.float64)
    wts = np.exp(wd) / np.exp(wd).sum()     # the fp32-rounded log weights, exactly
    expect = (wts[:, None] * v[0, 0, [0, 2, 3, 5]].double().numpy()).sum(axis=0)
    for h in range(Hq):
        np.testing.assert_allclose(out[0, 0, h], expect, rtol=0, atol=TIGHT)
