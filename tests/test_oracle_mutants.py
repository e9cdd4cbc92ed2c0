"""Plant plausible mistakes in copies of the C oracle; the pins must catch each.

Each mutant is a one-line textual change to ``oracle/fd_oracle.c`` compiled
into a temporary library (CPU only).  A battery of pins -- the hand-derived
fixtures, the float64 SDPA special case and the brute-force path -- runs
against it, and at least one pin must fail.  Mutants that would read outside
their buffers are deliberately not planted.
"""
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
from oracle import bruteforce
from decode_attention_preallocated_gb300 import workloads as W
from golden_cases import fixture_names, load as load_fixture
from test_oracle_pins import dense_mask, dq, gather_mask, sdpa_bias, sdpa_masked

SRC = os.path.join(os.path.dirname(oracle.__file__), "fd_oracle.c")

MUTANTS = {
    "drop_scale": ("score[t] = scale * dot +", "score[t] = dot +"),
    "bias_ignored": ("add[n] = (double)brow[t];", "add[n] = 0.0;"),
    "bias_negated": ("add[n] = (double)brow[t];", "add[n] = -(double)brow[t];"),
    "bias_neg_inf_kept": ("!(brow && isinf(brow[t]) && brow[t] < 0)", "1"),
    "causal_off_by_one": ("L - n_q + i : L - 1", "L - n_q + i - 1 : L - 1"),
    "causal_wrong_direction": ("L - n_q + i : L - 1", "L - 1 - i : L - 1"),
    "gqa_modulo_mapping": ("const int64_t hk = h / g;", "const int64_t hk = h % Hkv;"),
    "values_read_from_keys": ("orow[dd] += score[t] * kv_at(src, 1,",
                              "orow[dd] += score[t] * kv_at(src, 0,"),
    "no_normalisation": ("orow[dd] /= den;", "orow[dd] /= 1.0;"),
    "int8_scale_ignored": ("return (double)p[off] * s;", "return (double)p[off];"),
    "gather_drops_cell_zero": ("list[t] >= 0 &&", "list[t] >= 1 &&"),
    "bf16_widening": ("(uint32_t)bits << 16", "(uint32_t)bits << 15"),
    "row_index_swap": ("const int64_t i = (r / Hq) % n_q;",
                       "const int64_t i = r % n_q;"),
    "softmax_without_exp": ("score[t] = exp(score[t] - mx);",
                            "score[t] = score[t] - mx + 50.0;"),
}


def build_mutant(name, tmpdir):
    before, after = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(before) == 1, name
    path_c = os.path.join(tmpdir, name + ".c")
    path_so = os.path.join(tmpdir, name + ".so")
    with open(path_c, "w") as f:
        f.write(src.replace(before, after))
    subprocess.run(["gcc", "-O1", "-fPIC", "-shared", "-fopenmp", "-std=c99",
                    "-o", path_so, path_c, "-lm"], check=True)
    return oracle.load_variant(path_so)


def gather_bias_values(idx, seed):
    """Seeded per-cell biases for a gather list: N(0, 2), a few -inf, and one
    row that is -inf throughout."""
    g = torch.Generator().manual_seed(seed)
    bias = torch.randn(idx.shape, generator=g) * 2.0
    bias[0, 0, 1] = -float("inf")
    bias[-1, -1, 3] = -float("inf")
    bias[0, -1, :] = -float("inf")
    return bias


def battery(lib):
    """Run the pins against ``lib``; return the names of the pins that fail."""
    failed = []
    for name in fixture_names():
        fx = load_fixture(name)
        if fx["mode"] == "gather":
            out = lib.gather(fx["q"], fx["k"], fx["v"], fx["idx"], fx["scale"])
        else:
            out = lib.dense(fx["q"], fx["k"], fx["v"], fx["kv_lengths"], fx["n_q"],
                            fx["causal"], fx["scale"], fx["k_scale"], fx["v_scale"])
        if not np.allclose(out, fx["expected"].numpy(), rtol=0, atol=1e-12):
            failed.append("golden:" + name)
    for causal in (False, True):
        for int8 in (False, True):
            lens = (9, 14, 3)
            inp = W.dense_inputs(3, 3, 6, 2, 16, 16, list(lens), 5, causal,
                                 int8=int8)
            out = lib.dense(inp.q, inp.k, inp.v, inp.kv_lengths, 3, causal,
                            inp.scale, inp.k_scale, inp.v_scale)
            ref = sdpa_masked(inp.q.double(), dq(inp.k, inp.k_scale),
                              dq(inp.v, inp.v_scale),
                              dense_mask(lens, 3, 16, causal), inp.scale)
            if not np.allclose(out, ref.numpy(), rtol=0, atol=1e-12):
                failed.append("sdpa_dense(causal=%s,int8=%s)" % (causal, int8))
    inp = W.gather_inputs(2, 2, 8, 2, 16, 40, 12, 4, seed=9)
    out = lib.gather(inp.q, inp.k, inp.v, inp.idx, inp.scale)
    ref = sdpa_masked(inp.q.double(), inp.k.double(), inp.v.double(),
                      gather_mask(inp.idx, 40), inp.scale)
    if not np.allclose(out, ref.numpy(), rtol=0, atol=1e-12):
        failed.append("sdpa_gather")
    bias = gather_bias_values(inp.idx, 10)
    out = lib.gather(inp.q, inp.k, inp.v, inp.idx, inp.scale, bias=bias)
    ref = sdpa_bias(inp.q.double(), inp.k.double(), inp.v.double(), inp.idx, bias, 40,
                    inp.scale)
    if not np.allclose(out, ref.numpy(), rtol=0, atol=1e-12):
        failed.append("sdpa_gather_bias")
    inp = W.dense_inputs(2, 2, 4, 2, 4, 9, [6, 9], 11, True)
    out = lib.dense(inp.q, inp.k, inp.v, inp.kv_lengths, 2, True, inp.scale)
    ref = bruteforce.attend(inp.q.double().tolist(), inp.k.double().tolist(),
                            inp.v.double().tolist(),
                            lambda b, i: bruteforce.visible_dense([6, 9][b], 9, 2, i, True),
                            inp.scale)
    if not np.allclose(out, np.array(ref), rtol=0, atol=1e-12):
        failed.append("bruteforce")
    return failed


def test_unmutated_oracle_passes_battery(tmp_path):
    assert battery(oracle) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    lib = build_mutant(name, str(tmp_path))
    failed = battery(lib)
    assert failed, "mutant %s passed every pin" % name
