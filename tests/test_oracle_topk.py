"""Pins for the block top-k oracle (no GPU): a brute force with Python's
sorted() on small inputs, closed forms (every candidate selected gives the
prefix 0..L-1; strictly decreasing scores select the first blocks, strictly
increasing ones the last candidates; equal scores select the lowest
indices), and invariances (adding a constant or scaling by a positive
factor selects the same blocks)."""
import numpy as np
import pytest
import torch

import oracle


def brute(scores, lens, bs, k):
    B, n_q, nb = scores.shape
    out = np.full((B, n_q, k * bs), -1, dtype=np.int32)
    for b in range(B):
        L = min(max(int(lens[b]), 0), nb * bs)
        cands = [j for j in range(nb) if j * bs < L]
        for i in range(n_q):
            ranked = sorted(cands, key=lambda j: (-float(scores[b, i, j]), j))
            win = sorted(ranked[:k])
            cells = []
            for j in win:
                for c in range(bs):
                    x = j * bs + c
                    cells.append(x if x < L else -1)
            out[b, i, :len(cells)] = cells
    return out


@pytest.mark.parametrize("seed", range(6))
def test_matches_bruteforce(seed):
    g = torch.Generator().manual_seed(seed)
    B, n_q, nb = 3, 2, 37
    bs, k = 1 + seed % 4, 1 + (seed * 5) % 11
    scores = torch.randn(B, n_q, nb, generator=g)
    scores[0, 0, 3] = scores[0, 0, 9]                    # a tie
    scores[1, 1, :5] = -float("inf")
    scores[2, 0, 7] = -0.0
    scores[2, 0, 8] = 0.0
    lens = [nb * bs, 0, 17]
    got = oracle.topk_blocks(scores, torch.tensor(lens, dtype=torch.int32), bs, k)
    np.testing.assert_array_equal(got, brute(scores.numpy(), lens, bs, k))


def test_every_candidate_selected_gives_the_prefix():
    scores = torch.randn(2, 3, 20, generator=torch.Generator().manual_seed(7))
    lens = torch.tensor([45, 80], dtype=torch.int32)
    got = oracle.topk_blocks(scores, lens, 4, 20)
    for b, L in enumerate([45, 80]):
        for i in range(3):
            want = list(range(L)) + [-1] * (80 - L)
            assert got[b, i].tolist() == want


def test_monotone_and_equal_scores():
    nb, bs, k = 16, 2, 5
    dec = torch.arange(nb, 0, -1, dtype=torch.float32).view(1, 1, nb)
    inc = torch.arange(nb, dtype=torch.float32).view(1, 1, nb)
    eq = torch.full((1, 1, nb), 3.5)
    L = torch.tensor([29], dtype=torch.int32)            # 15 candidates, the last one partial
    first = [c for j in range(5) for c in (2 * j, 2 * j + 1)]
    assert oracle.topk_blocks(dec, L, bs, k)[0, 0].tolist() == first
    assert oracle.topk_blocks(eq, L, bs, k)[0, 0].tolist() == first
    last = [c if c < 29 else -1 for j in range(10, 15) for c in (2 * j, 2 * j + 1)]
    assert oracle.topk_blocks(inc, L, bs, k)[0, 0].tolist() == last


def test_shift_and_positive_scale_do_not_change_the_selection():
    g = torch.Generator().manual_seed(8)
    scores = torch.randn(2, 2, 50, generator=g)
    lens = torch.tensor([400, 123], dtype=torch.int32)
    a = oracle.topk_blocks(scores, lens, 8, 7)
    b = oracle.topk_blocks(scores * 4.0 + 100.0, lens, 8, 7)
    np.testing.assert_array_equal(a, b)
