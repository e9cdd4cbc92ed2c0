"""Pins for the fp64 CPU oracle (no GPU).

Each test ties ``oracle.dense`` / ``oracle.gather`` to something other than
the oracle itself: closed forms, the hand-derived fixtures, a library routine
(torch SDPA in float64 with an explicit mask), a second brute-force path, and
the invariants the pages state or imply.  ``test_oracle_mutants.py`` checks
that planted mistakes in the C oracle fail this suite.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import bruteforce
from decode_attention_preallocated_gb300 import workloads as W
from golden_cases import fixture_names, load as load_fixture

TIGHT = 1e-12


# ----------------------------------------------------------------- helpers
def dq(x, scale=None):
    """Dequantised float64 view of a cache (bf16 or int8 * per-token scale)."""
    if x.dtype == torch.int8:
        return x.double() * scale.double().unsqueeze(-1)
    return x.double()


def sdpa_masked(q, k, v, mask, scale):
    """torch SDPA in float64: q [B,n_q,Hq,d], k/v [B,Hkv,cap,d] float64,
    mask [B,n_q,cap] bool (True = visible).  Rows with nothing visible -> 0."""
    B, n_q, Hq, d = q.shape
    g = Hq // k.shape[1]
    kk = k.repeat_interleave(g, dim=1)
    vv = v.repeat_interleave(g, dim=1)
    qq = q.permute(0, 2, 1, 3)
    m = mask[:, None, :, :].expand(B, Hq, n_q, k.shape[2])
    out = F.scaled_dot_product_attention(qq, kk, vv, attn_mask=m, scale=scale)
    out = out.permute(0, 2, 1, 3).contiguous()
    empty = ~mask.any(dim=-1)                       # [B, n_q]
    out[empty[:, :, None, None].expand_as(out)] = 0.0
    return out


def sdpa_bias(q, k, v, idx, bias, cap, scale):
    """torch SDPA in float64 with an additive float mask built from a gather
    list and its per-cell biases (cells not listed, out of range or -inf are
    -inf); rows with nothing visible -> 0.  idx must list distinct cells."""
    B, n_q, K = idx.shape
    m = torch.full((B, n_q, cap), -float("inf"), dtype=torch.float64)
    for b in range(B):
        for i in range(n_q):
            for t, j in enumerate(idx[b, i].tolist()):
                if 0 <= j < cap:
                    m[b, i, j] = float(bias[b, i, t])
    g = q.shape[2] // k.shape[1]
    kk = k.repeat_interleave(g, dim=1)
    vv = v.repeat_interleave(g, dim=1)
    qq = q.permute(0, 2, 1, 3)
    visible = torch.isfinite(m)
    safe = torch.where(visible, m, torch.full_like(m, -1e300))
    mm = safe[:, None, :, :].expand(B, q.shape[2], n_q, cap)
    out = F.scaled_dot_product_attention(qq, kk, vv, attn_mask=mm, scale=scale)
    out = out.permute(0, 2, 1, 3).contiguous()
    empty = ~visible.any(dim=-1)
    out[empty[:, :, None, None].expand_as(out)] = 0.0
    return out


def dense_mask(lengths, n_q, cap, causal):
    """Visible-key mask built from the definition by hand."""
    B = len(lengths)
    m = torch.zeros(B, n_q, cap, dtype=torch.bool)
    for b, L in enumerate(lengths):
        L = max(0, min(int(L), cap))
        for i in range(n_q):
            last = L - n_q + i if causal else L - 1
            if last >= 0:
                m[b, i, : last + 1] = True
    return m


def gather_mask(idx, cap):
    B, n_q, K = idx.shape
    m = torch.zeros(B, n_q, cap, dtype=torch.bool)
    for b in range(B):
        for i in range(n_q):
            for j in idx[b, i].tolist():
                if 0 <= j < cap:
                    m[b, i, j] = True
    return m


def small_dense(seed, B=2, n_q=3, Hq=4, Hkv=2, d=8, cap=12, lengths=(7, 12),
                causal=True, int8=False, layout="bhtd", tail="randn"):
    return W.dense_inputs(B, n_q, Hq, Hkv, d, cap, list(lengths), seed, causal,
                          layout=layout, tail=tail, int8=int8)


def run_dense(inp):
    return torch.from_numpy(oracle.dense(inp.q, inp.k, inp.v, inp.kv_lengths,
                                         inp.n_q, inp.causal, inp.scale,
                                         inp.k_scale, inp.v_scale))


# ------------------------------------------------------------ fixtures
@pytest.mark.parametrize("name", fixture_names())
def test_golden_fixture(name):
    fx = load_fixture(name)
    if fx["mode"] == "gather":
        out = oracle.gather(fx["q"], fx["k"], fx["v"], fx["idx"], fx["scale"])
    else:
        out = oracle.dense(fx["q"], fx["k"], fx["v"], fx["kv_lengths"],
                           fx["n_q"], fx["causal"], fx["scale"],
                           fx["k_scale"], fx["v_scale"])
    np.testing.assert_allclose(out, fx["expected"].numpy(), rtol=0, atol=1e-14)


# ---------------------------------------------------------- closed forms
def test_single_key_returns_its_value_row():
    inp = small_dense(3, n_q=1, lengths=(1, 1), causal=False)
    out = run_dense(inp)
    g = 2
    for b in range(2):
        for h in range(4):
            assert torch.equal(out[b, 0, h], inp.v[b, h // g, 0].double())


def test_identical_keys_give_mean_of_visible_values():
    inp = small_dense(4, n_q=2, lengths=(5, 9), causal=True)
    inp.k[:] = inp.k[:, :, :1, :]          # every position holds the same key
    out = run_dense(inp)
    for b, L in enumerate((5, 9)):
        for i in range(2):
            last = L - 2 + i
            for h in range(4):
                mean = inp.v[b, h // 2, : last + 1].double().mean(0)
                torch.testing.assert_close(out[b, i, h], mean, rtol=0, atol=1e-14)


def test_constant_values_are_returned():
    inp = small_dense(5, causal=False)
    inp.v.fill_(1.5)
    out = run_dense(inp)
    assert torch.allclose(out, torch.full_like(out, 1.5), rtol=0, atol=1e-14)


def test_zero_query_is_uniform_mean():
    inp = small_dense(6, causal=False)
    inp.q.zero_()
    out = run_dense(inp)
    for b, L in enumerate((7, 12)):
        for h in range(4):
            mean = inp.v[b, h // 2, :L].double().mean(0)
            torch.testing.assert_close(out[b, 0, h], mean, rtol=0, atol=1e-14)


def test_dominant_key_returns_its_row():
    # all other keys are zero (score 0) and key j scores >= 40, so every other
    # weight is below e^-40 relative to key j's
    inp = small_dense(7, n_q=1, Hq=2, Hkv=1, lengths=(10, 10), causal=False)
    j = 4
    keep = inp.k[:, :, j].clone()
    inp.k.zero_()
    inp.k[:, :, j] = keep
    for b in range(2):
        kj = inp.k[b, 0, j].double()
        c = 48.0 / (inp.scale * float(kj @ kj))
        inp.q[b, 0, :] = (c * kj).to(torch.bfloat16)
        s = inp.scale * float(inp.q[b, 0, 0].double() @ kj)
        assert s > 40
    out = run_dense(inp)
    for b in range(2):
        for h in range(2):
            torch.testing.assert_close(out[b, 0, h], inp.v[b, 0, j].double(),
                                       rtol=0, atol=1e-12)


def test_empty_visible_set_gives_zeros():
    # L = 0, and causal rows whose window starts before position 0
    inp = small_dense(8, n_q=3, lengths=(0, 1), causal=True)
    out = run_dense(inp)
    assert torch.count_nonzero(out[0]) == 0
    assert torch.count_nonzero(out[1, 0]) == 0 and torch.count_nonzero(out[1, 1]) == 0
    for h in range(4):
        assert torch.equal(out[1, 2, h], inp.v[1, h // 2, 0].double())


# ------------------------------------------------------ library special case
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n_q", [1, 2, 6])
@pytest.mark.parametrize("int8", [False, True])
def test_matches_sdpa_float64_dense(causal, n_q, int8):
    lengths = (9, 14, 3)
    inp = small_dense(10 + n_q, B=3, n_q=n_q, Hq=6, Hkv=2, d=16, cap=16,
                      lengths=lengths, causal=causal, int8=int8)
    out = run_dense(inp)
    ref = sdpa_masked(inp.q.double(), dq(inp.k, inp.k_scale), dq(inp.v, inp.v_scale),
                      dense_mask(lengths, n_q, 16, causal), inp.scale)
    torch.testing.assert_close(out, ref, rtol=0, atol=TIGHT)


def test_matches_sdpa_float64_gather():
    inp = W.gather_inputs(2, 3, 8, 2, 16, 40, 12, 4, seed=21)
    idx = inp.idx.clone()
    idx[0, 1, 3] = -1                 # padding
    idx[1, 2, 5] = 40                 # past the capacity: skipped
    out = torch.from_numpy(oracle.gather(inp.q, inp.k, inp.v, idx, inp.scale))
    ref = sdpa_masked(inp.q.double(), inp.k.double(), inp.v.double(),
                      gather_mask(idx, 40), inp.scale)
    torch.testing.assert_close(out, ref, rtol=0, atol=TIGHT)


# ------------------------------------------------------------- brute force
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("int8", [False, True])
def test_matches_bruteforce_dense(causal, int8):
    lengths = (6, 11)
    inp = small_dense(30, B=2, n_q=3, Hq=4, Hkv=2, d=4, cap=11, lengths=lengths,
                      causal=causal, int8=int8)
    out = run_dense(inp)
    qf = inp.q.double().tolist()
    kf = dq(inp.k, inp.k_scale).tolist()
    vf = dq(inp.v, inp.v_scale).tolist()
    ref = bruteforce.attend(
        qf, kf, vf,
        lambda b, i: bruteforce.visible_dense(lengths[b], 11, 3, i, causal),
        inp.scale)
    np.testing.assert_allclose(out.numpy(), np.array(ref), rtol=0, atol=TIGHT)


def test_matches_bruteforce_gather():
    inp = W.gather_inputs(2, 2, 4, 2, 8, 30, 9, 3, seed=31)
    idx = inp.idx.clone()
    idx[1, 0, 2] = -5
    idx[0, 1, 0] = 1000
    out = oracle.gather(inp.q, inp.k, inp.v, idx, inp.scale)
    ref = bruteforce.attend(
        inp.q.double().tolist(), inp.k.double().tolist(), inp.v.double().tolist(),
        lambda b, i: bruteforce.visible_gather(idx[b, i].tolist(), 30), inp.scale)
    np.testing.assert_allclose(out, np.array(ref), rtol=0, atol=TIGHT)


# ---------------------------------------------------------------- invariants
def test_gather_of_prefix_equals_dense():
    L, cap = 13, 20
    inp = small_dense(40, B=1, n_q=1, cap=cap, lengths=(L,), causal=False)
    dense = run_dense(inp)
    idx = torch.arange(L, dtype=torch.int32).view(1, 1, L)
    g = oracle.gather(inp.q, inp.k, inp.v, idx, inp.scale)
    np.testing.assert_array_equal(g, dense.numpy())
    perm = idx[:, :, torch.randperm(L, generator=torch.Generator().manual_seed(1))]
    g2 = oracle.gather(inp.q, inp.k, inp.v, perm, inp.scale)
    np.testing.assert_allclose(g2, dense.numpy(), rtol=0, atol=TIGHT)


def test_gather_selection_equals_masked_dense_and_is_order_free():
    inp = W.gather_inputs(1, 2, 8, 2, 16, 64, 10, 2, seed=41)
    a = oracle.gather(inp.q, inp.k, inp.v, inp.idx, inp.scale)
    shuffled = inp.idx[:, :, torch.randperm(10, generator=torch.Generator().manual_seed(2))]
    b = oracle.gather(inp.q, inp.k, inp.v, shuffled, inp.scale)
    np.testing.assert_allclose(a, b, rtol=0, atol=TIGHT)
    ref = sdpa_masked(inp.q.double(), inp.k.double(), inp.v.double(),
                      gather_mask(inp.idx, 64), inp.scale)
    np.testing.assert_allclose(a, ref.numpy(), rtol=0, atol=TIGHT)


def test_capacity_and_tail_do_not_matter():
    lengths = (9, 5)
    a = small_dense(50, cap=9, lengths=lengths)
    big = small_dense(51, cap=40, lengths=lengths, tail="nan")
    big.q.copy_(a.q)
    big.k[:, :, :9] = a.k
    big.v[:, :, :9] = a.v
    out_a, out_b = run_dense(a), run_dense(big)
    assert torch.equal(out_a, out_b)
    assert torch.isfinite(out_b).all()


def test_token_major_layout_matches_canonical():
    a = small_dense(52, layout="bhtd")
    b = small_dense(52, layout="bthd")
    assert b.k.stride(2) != 8 and b.k.stride(1) == 8
    b.k.copy_(a.k)
    b.v.copy_(a.v)
    b.q.copy_(a.q)
    assert torch.equal(run_dense(a), run_dense(b))


def test_causal_row_ignores_later_drafts():
    n_q, L = 4, 10
    a = small_dense(60, B=1, n_q=n_q, cap=12, lengths=(L,), causal=True)
    out_a = run_dense(a)
    for i in range(n_q - 1):
        b = small_dense(60, B=1, n_q=n_q, cap=12, lengths=(L,), causal=True)
        first_hidden = L - n_q + i + 1
        b.k[:, :, first_hidden:L] = 3.0
        b.v[:, :, first_hidden:L] = -7.0
        out_b = run_dense(b)
        assert torch.equal(out_a[0, : i + 1], out_b[0, : i + 1])
        assert not torch.equal(out_a[0, i + 1:], out_b[0, i + 1:])


def test_single_row_causal_equals_noncausal():
    a = small_dense(61, n_q=1, causal=True)
    b = small_dense(61, n_q=1, causal=False)
    assert torch.equal(run_dense(a), run_dense(b))


def test_rollback_by_length():
    inp = small_dense(62, B=1, n_q=2, cap=20, lengths=(15,), causal=True)
    fresh = small_dense(62, B=1, n_q=2, cap=20, lengths=(12,), causal=True)
    # decode at 15 with three accepted drafts, then roll back to 12
    _ = run_dense(inp)
    inp.kv_lengths[0] = 12
    rolled = oracle.dense(inp.q, inp.k, inp.v, [12], 2, True, inp.scale)
    np.testing.assert_array_equal(rolled, run_dense(fresh).numpy())


def test_lengths_are_clamped_to_capacity():
    inp = small_dense(63, lengths=(-4, 99), causal=False)
    out = run_dense(inp)
    assert torch.count_nonzero(out[0]) == 0
    full = oracle.dense(inp.q, inp.k, inp.v, [0, 12], 3, False, inp.scale)
    np.testing.assert_array_equal(out.numpy(), full)


def test_int8_oracle_equals_bf16_oracle_on_dequantised_values():
    # fixed-point codes * power-of-two scales are bf16-exact, so the int8
    # widening must agree with the bf16 path bit for bit
    g = torch.Generator().manual_seed(70)
    B, Hkv, cap, d = 1, 2, 10, 8
    codes_k = torch.randint(-127, 128, (B, Hkv, cap, d), generator=g).to(torch.int8)
    codes_v = torch.randint(-127, 128, (B, Hkv, cap, d), generator=g).to(torch.int8)
    sk = 2.0 ** torch.randint(-9, -3, (B, Hkv, cap), generator=g).float()
    sv = 2.0 ** torch.randint(-9, -3, (B, Hkv, cap), generator=g).float()
    kb = (codes_k.double() * sk.double()[..., None]).to(torch.bfloat16)
    vb = (codes_v.double() * sv.double()[..., None]).to(torch.bfloat16)
    assert torch.equal(kb.double(), codes_k.double() * sk.double()[..., None])
    q = W.randn_bf16((B, 2, 4, d), g, "cpu")
    a = oracle.dense(q, codes_k, codes_v, [8], 2, True, 0.3, sk, sv)
    b = oracle.dense(q, kb, vb, [8], 2, True, 0.3)
    np.testing.assert_array_equal(a, b)


def test_workload_recipes_have_the_stated_shapes():
    r = W.ragged_lengths(8, 1024, 32768, 1)
    assert len(r) == 8 and all(1024 <= x <= 32768 for x in r)
    g = torch.Generator().manual_seed(3)
    idx = W.topk_like_indices(1000, 64, 8, g, 3)
    for row in idx:
        s = set(row.tolist())
        assert len(s) == 64 and set(range(992, 1000)) <= s
        assert all(0 <= x < 1000 for x in s)
    x = torch.randn(2, 3, 5, 16, generator=g)
    codes, scale = W.quantize_per_token(x)
    assert codes.abs().max() <= 127
    err = (codes.double() * scale.double()[..., None] - x.double()).abs()
    assert (err <= scale.double()[..., None] / 2 + 1e-7).all()
