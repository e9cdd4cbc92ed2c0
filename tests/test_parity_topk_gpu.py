"""GPU parity of the block top-k selection (fd_topk_blocks) against the
oracle, bit for bit: block counts from 1 to the 32768 limit, block sizes 1
to 64, top_k below, at and above the candidate count, lengths 0, partial
blocks and past the span, ties, -inf and signed zeros; then the whole
selection + gather step against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from decode_attention_preallocated_gb300 import build as fdbuild
from decode_attention_preallocated_gb300 import fd
from decode_attention_preallocated_gb300 import workloads as W
from parity_util import compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    fdbuild.build()
    fd.lib()


def scores_for(B, n_q, nb, seed, ties=True):
    g = torch.Generator().manual_seed(seed)
    s = torch.randn(B, n_q, nb, generator=g)
    if ties and nb > 8:
        # coarse values make many ties; a few -inf and signed zeros
        s[0] = torch.round(s[0] * 2.0) / 2.0
        s[-1, -1, 1::7] = -float("inf")
        s[0, 0, 2] = -0.0
        s[0, 0, 5] = 0.0
    return s


CASES = [
    # B, n_q, n_blocks, block_size, top_k, lengths
    (1, 1, 1, 1, 1, [1]),
    (2, 3, 37, 4, 5, [148, 61]),
    (3, 2, 2048, 64, 32, [131072, 0, 70001]),
    (1, 4, 2048, 1, 2048, [1500]),
    (2, 1, 500, 16, 600, [8000, 7999]),
    (8, 6, 512, 64, 32, [32768, 1024, 5000, 64, 65, 12000, 32767, 900000]),
    (1, 2, 32768, 8, 257, [262144]),
    (2, 2, 30000, 3, 1000, [45000, 90000]),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_topk_matches_oracle(case):
    B, n_q, nb, bs, k, lens = CASES[case]
    s = scores_for(B, n_q, nb, 70 + case)
    lens_t = torch.tensor(lens, dtype=torch.int32)
    ref = oracle.topk_blocks(s, lens_t, bs, k)
    got = fd.topk_blocks(s.cuda(), lens_t.cuda(), bs, k)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(got.cpu().numpy(), ref)


def test_topk_rejects_too_many_blocks():
    s = torch.zeros(1, 1, 32769, device="cuda")
    with pytest.raises(fd.FdError):
        fd.topk_blocks(s, torch.tensor([10], dtype=torch.int32, device="cuda"), 1, 1)


def test_select_then_gather_matches_oracle():
    # block scores -> lists -> gather attention, both on the GPU, against the
    # oracle's lists and the oracle's gather
    B, n_q, Hq, Hkv, d, cap, bs, k = 2, 2, 16, 4, 128, 20000, 64, 24
    nb = cap // bs + 1
    inp = W.dense_inputs(B, n_q, Hq, Hkv, d, nb * bs, [19000, 7321], 80, False)
    s = scores_for(B, n_q, nb, 81, ties=False)
    lens = inp.kv_lengths
    ref_idx = oracle.topk_blocks(s, lens, bs, k)
    ref = oracle.gather(inp.q, inp.k, inp.v, torch.from_numpy(ref_idx), inp.scale)
    idx = fd.topk_blocks(s.cuda(), lens.cuda(), bs, k)
    out = fd.decode_gather(inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), idx, scale=inp.scale,
                           out_dtype=torch.float32)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx)
    compare(out, torch.from_numpy(ref), torch.float32, "select + gather")
