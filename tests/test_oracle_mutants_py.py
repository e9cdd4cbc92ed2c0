"""Plant plausible mistakes in copies of the Python-level oracle functions
(paged cache, fused append, masked prefix, block top-k); the pins must
catch each.

Each mutant is a one-line textual change to ``oracle/__init__.py``, loaded
as a separate module from a temporary copy of the package (CPU only).  A
battery of the pins of that function runs against it -- float64 SDPA over
other constructions, the sorted() brute force, the cache state after an
append -- and at least one must fail (an exception counts as a failure).
"""
import importlib.util
import os
import shutil

import numpy as np
import pytest
import torch

import oracle
from decode_attention_preallocated_gb300 import workloads as W
from test_oracle_append import concat_reference, new_rows
from test_oracle_masked import sdpa_additive
from test_oracle_paged import paged_from_flat
from test_oracle_pins import TIGHT, dense_mask, dq, sdpa_masked
from test_oracle_topk import brute

SRC_DIR = os.path.dirname(oracle.__file__)

MUTANTS = {
    # paged cache
    "paged_page_from_row": ("page = table[:, j // ps]", "page = table[:, j % ps]"),
    "paged_row_from_page": ("row = np.broadcast_to(j % ps, pg.shape)",
                            "row = np.broadcast_to(j // ps % ps, pg.shape)"),
    "paged_bad_entries_kept": ("on_pool = (page >= 0) & (page < P)",
                               "on_pool = page < P"),
    # fused append
    "append_one_past": ("pos = int(base[b]) + i", "pos = int(base[b]) + i + 1"),
    "append_rows_reversed": ("ka[b, :, pos, :] = kn[b, i]", "ka[b, :, pos, :] = kn[b, n - 1 - i]"),
    "append_length_not_advanced": ("after = np.minimum(base + n, cap).astype(np.int32)",
                                   "after = np.minimum(base + n - 1, cap).astype(np.int32)"),
    # masked prefix
    "masked_bias_dropped": ("bias[r, :len(cells)] = ma[r // n_q, r % n_q, cells]",
                            "bias[r, :len(cells)] = 0.0"),
    "masked_window_off_by_one": ("            last = L - n_q + i if causal else L - 1\n            cells = np.arange",
                                 "            last = L - n_q + i - 1 if causal else L - 1\n            cells = np.arange"),
    # block top-k
    "topk_ties_to_higher_index": ("order = np.lexsort((cand, -s))", "order = np.lexsort((-cand, -s))"),
    "topk_winners_unsorted": ("chosen = np.sort(order[:top_k])", "chosen = order[:top_k]"),
    "topk_partial_block_dropped": ("nvalid = min(nb, -(-L // block_size))",
                                   "nvalid = min(nb, L // block_size)"),
}


def load_mutant(name, tmp_path):
    before, after = MUTANTS[name]
    pkg = tmp_path / ("oracle_" + name)
    pkg.mkdir()
    src = open(os.path.join(SRC_DIR, "__init__.py")).read()
    assert src.count(before) == 1, name
    (pkg / "__init__.py").write_text(src.replace(before, after))
    for f in ("fd_oracle.c", "liboracle.so", "bruteforce.py"):
        shutil.copy2(os.path.join(SRC_DIR, f), pkg / f)
    spec = importlib.util.spec_from_file_location("oracle_" + name, pkg / "__init__.py",
                                                  submodule_search_locations=[str(pkg)])
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def battery_paged(lib):
    cap = 24
    for ps, causal in ((3, True), (4, False)):
        inp = W.dense_inputs(3, 3, 6, 2, 16, cap, [19, 24, 5], 40 + ps, causal)
        kp, vp, _, _, table = paged_from_flat(inp, ps, 7 + ps)
        out = lib.paged(inp.q, kp, vp, table, inp.kv_lengths, 3, causal, inp.scale)
        ref = sdpa_masked(inp.q.double(), inp.k.double(), inp.v.double(),
                          dense_mask([19, 24, 5], 3, cap, causal), inp.scale)
        if not np.allclose(out, ref.numpy(), rtol=0, atol=TIGHT):
            return True
    inp = W.dense_inputs(2, 2, 4, 2, 8, cap, [22, 17], 51, True)
    kp, vp, _, _, table = paged_from_flat(inp, 4, 52)
    table = table.clone()
    table[0, 2] = -1
    out = lib.paged(inp.q, kp, vp, table, inp.kv_lengths, 2, True, inp.scale)
    m = dense_mask([22, 17], 2, cap, True)
    m[0, :, 8:12] = False
    ref = sdpa_masked(inp.q.double(), inp.k.double(), inp.v.double(), m, inp.scale)
    return not np.allclose(out, ref.numpy(), rtol=0, atol=TIGHT)


def battery_append(lib):
    inp = W.dense_inputs(2, 3, 6, 2, 16, 40, [17, 33], 93, True)
    kn, vn = new_rows(2, 3, 2, 16, 94)
    out, ka, _, after = lib.append(inp.q, inp.k, inp.v, kn, vn, inp.kv_lengths, True, inp.scale)
    if after.tolist() != [20, 36]:
        return True
    knb = kn.view(torch.int16).numpy().view(np.uint16)
    for b, L in enumerate([17, 33]):
        for i in range(3):
            if not np.array_equal(ka[b, :, L + i], knb[b, i]):
                return True
    ref = concat_reference(inp, kn, vn, True)
    return not np.allclose(out, ref.numpy(), rtol=0, atol=TIGHT)


def battery_masked(lib):
    cap = 96
    for n_q, causal in ((3, True), (1, False)):
        inp = W.dense_inputs(3, n_q, 6, 2, 16, cap, [90, 0, 41], 110 + n_q, causal)
        g = torch.Generator().manual_seed(111)
        mask = torch.randn(3, n_q, cap, generator=g) * 2.0
        mask[torch.rand(3, n_q, cap, generator=g) < 0.5] = -float("inf")
        out = lib.masked(inp.q, inp.k, inp.v, inp.kv_lengths, mask, n_q, causal, inp.scale)
        if not np.allclose(out, sdpa_additive(inp, mask, causal).numpy(), rtol=0, atol=TIGHT):
            return True
    return False


def battery_topk(lib):
    for seed in range(4):
        g = torch.Generator().manual_seed(seed)
        scores = torch.round(torch.randn(3, 2, 37, generator=g) * 2.0) / 2.0   # many ties
        lens = [37 * 3, 0, 17]
        bs, k = 3, 1 + (seed * 5) % 11
        got = lib.topk_blocks(scores, torch.tensor(lens, dtype=torch.int32), bs, k)
        if not np.array_equal(got, brute(scores.numpy(), lens, bs, k)):
            return True
    return False


BATTERY = {"paged": battery_paged, "append": battery_append, "masked": battery_masked,
           "topk": battery_topk}


def fails(battery, lib):
    try:
        return battery(lib)
    except Exception:
        return True


def test_unmutated_oracle_passes_every_battery():
    for name, battery in BATTERY.items():
        assert not fails(battery, oracle), name


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    lib = load_mutant(name, tmp_path)
    battery = BATTERY[name.split("_")[0]]
    assert fails(battery, lib), "mutant %s passed every pin" % name
