"""GPU parity of the masked prefix with chunk skipping (fd_decode_masked)
against the fp64 oracle, on the CUDA-core kernel and on the tensor-core
kernel both with its chunk list (the default workspace has room for it) and
with chunks found in place (a workspace sized for the call alone): masks
that hide most 32-position chunks, seeded finite biases, causal windows,
ragged and empty sequences, NaN past the lengths, head_dim 128 and 256,
split counts, everything hidden, lists longer than one listing block,
consecutive calls with other masks, graph replay, and the mask built from
the gather workload's list."""
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


def chunk_mask(B, n_q, cap, seed, keep=0.15):
    """N(0, 2) biases on a random ~keep share of 32-position chunks (and on
    a few single cells elsewhere), -inf on the rest."""
    g = torch.Generator().manual_seed(seed)
    m = torch.full((B, n_q, cap), -float("inf"))
    nch = (cap + 31) // 32
    live = torch.rand(B, nch, generator=g) < keep
    for b in range(B):
        for c in torch.nonzero(live[b]).flatten().tolist():
            m[b, :, c * 32:(c + 1) * 32] = torch.randn(n_q, min(32, cap - c * 32), generator=g) * 2
    cells = torch.randint(0, cap, (B, 8), generator=g)
    for b in range(B):
        m[b, 0, cells[b]] = 0.5
    return m


# "tc" has room for the chunk list; "tc_in_place" gets a workspace of exactly
# the call's segments, rows, head_dim and blocks, which leaves none
KERNELS = ["simt", "tc", "tc_in_place"]
IN_PLACE_CTAS = 148


def rows_of(inp):
    return inp.q.shape[2] // inp.k.shape[1] * inp.n_q


def make_ws(inp, kernel):
    nseg = inp.q.shape[0] * inp.k.shape[1]
    if kernel == "tc_in_place":
        return fd.Workspace(nseg, rows_of(inp), inp.q.shape[3], IN_PLACE_CTAS)
    return fd.Workspace(nseg, 64, 256, 2048)


def run(inp, mask, out_dtype, num_ctas=0, kernel="tc", ws=None):
    own = ws is None
    ws = make_ws(inp, kernel) if own else ws
    if kernel == "tc_in_place":
        num_ctas = num_ctas or IN_PLACE_CTAS
        assert ws.max_ctas == num_ctas
    kid = fd.FD_KERNEL_SIMT if kernel == "simt" else fd.FD_KERNEL_TC
    out = fd.decode_masked(inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), inp.kv_lengths.cuda(),
                           mask.cuda(), n_q=inp.n_q, causal=inp.causal, scale=inp.scale,
                           out_dtype=out_dtype, num_ctas=num_ctas, kernel=kid, workspace=ws)
    torch.cuda.synchronize()
    assert not ws.diagnostics()[0] & fd.FD_DEV_INTERNAL
    if own:
        ws.close()
    return out

CASES = {
    "d128_decode": (3, 1, 8, 2, 128, 3000, [3000, 1, 1777], False),
    "d256_mtp": (2, 4, 16, 4, 256, 2500, [2500, 999], True),
    "d256_ragged6": (3, 6, 16, 4, 256, 1400, [1400, 263, 1291], True),
    "rows48": (2, 3, 64, 4, 128, 900, [900, 77], True),
    "rows64": (2, 2, 32, 1, 128, 1200, [1200, 0], True),
}


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("case", sorted(CASES))
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_masked_matches_oracle(case, out_dtype, kernel):
    B, n_q, Hq, Hkv, d, cap, lens, causal = CASES[case]
    # NaN past each length: a read of the tail would reach the output
    inp = W.dense_inputs(B, n_q, Hq, Hkv, d, cap, lens, 120, causal, tail="nan")
    mask = chunk_mask(B, n_q, cap, 121)
    ref = torch.from_numpy(oracle.masked(inp.q, inp.k, inp.v, inp.kv_lengths, mask, n_q,
                                         causal, inp.scale))
    compare(run(inp, mask, out_dtype, kernel=kernel), ref, out_dtype, case)


@pytest.mark.parametrize("kernel", ["simt", "tc"])
@pytest.mark.parametrize("ctas", [1, 7, 300])
def test_masked_split_counts_and_hidden_rows(ctas, kernel):
    inp = W.dense_inputs(2, 3, 8, 2, 256, 2000, [2000, 1500], 122, True)
    mask = chunk_mask(2, 3, 2000, 123, keep=0.3)
    mask[1, 2, :] = -float("inf")                       # a row with nothing visible
    ref = torch.from_numpy(oracle.masked(inp.q, inp.k, inp.v, inp.kv_lengths, mask, 3, True,
                                         inp.scale))
    got = run(inp, mask, torch.float32, num_ctas=ctas, kernel=kernel)
    compare(got, ref, torch.float32, "masked splits")
    assert torch.count_nonzero(got[1, 2].cpu()) == 0


@pytest.mark.parametrize("kernel", KERNELS)
def test_masked_everything_hidden_gives_zeros(kernel):
    inp = W.dense_inputs(2, 2, 8, 2, 128, 700, [700, 300], 124, True)
    mask = torch.full((2, 2, 700), -float("inf"))
    got = run(inp, mask, torch.float32, kernel=kernel)
    assert torch.count_nonzero(got.cpu()) == 0


@pytest.mark.parametrize("kernel", KERNELS)
def test_masked_from_a_gather_list(kernel):
    # the gather workload's selection as a mask over the whole window
    inp = W.gather_inputs(1, 1, 32, 4, 128, 131072, 2048, 128, seed=1)
    mask = torch.full((1, 1, 131072), -float("inf"))
    mask[0, 0, inp.idx[0, 0].long()] = 0.0
    dense = W.DecodeInputs(q=inp.q, k=inp.k, v=inp.v, kv_lengths=inp.kv_lengths, n_q=1,
                           causal=False, scale=inp.scale)
    ref = torch.from_numpy(oracle.gather(inp.q, inp.k, inp.v, inp.idx, inp.scale))
    for od in (torch.bfloat16, torch.float32):
        compare(run(dense, mask, od, kernel=kernel), ref, od, "masked = gather")


@pytest.mark.parametrize("kernel", ["tc", "tc_in_place"])
def test_masked_long_lists_several_listing_blocks(kernel):
    # 20000 positions = 625 chunks: three blocks of the listing pass per
    # sequence; lengths that end inside a chunk; a sequence whose only
    # visible chunks are its first and its (partial) last
    lens = [20000, 13001, 9999]
    inp = W.dense_inputs(3, 2, 16, 2, 128, 20000, lens, 130, True, tail="nan")
    mask = chunk_mask(3, 2, 20000, 131, keep=0.4)
    mask[2] = -float("inf")
    mask[2, :, 0:5] = 0.25
    mask[2, 1, 9990:9999] = -0.5
    ref = torch.from_numpy(oracle.masked(inp.q, inp.k, inp.v, inp.kv_lengths, mask, 2, True,
                                         inp.scale))
    for od in (torch.bfloat16, torch.float32):
        compare(run(inp, mask, od, kernel=kernel), ref, od, "long lists " + kernel)


def test_masked_consecutive_calls_share_a_workspace():
    # the listing pass's counters must be back at zero for the next call
    inp = W.dense_inputs(2, 1, 8, 2, 256, 6000, [6000, 4100], 132, False)
    ws = make_ws(inp, "tc")
    for seed, keep in ((133, 0.05), (134, 0.5), (135, 0.0), (136, 1.0)):
        mask = chunk_mask(2, 1, 6000, seed, keep=keep)
        ref = torch.from_numpy(oracle.masked(inp.q, inp.k, inp.v, inp.kv_lengths, mask, 1,
                                             False, inp.scale))
        compare(run(inp, mask, torch.float32, kernel="tc", ws=ws), ref, torch.float32,
                "call with keep %.2f" % keep)
    assert ws.device_status() == 0
    ws.close()


def test_masked_chunk_list_in_a_graph():
    # the listing pass and the decode replay from a graph, with the mask and
    # the lengths rewritten on the device between replays
    inp = W.dense_inputs(2, 2, 16, 4, 128, 8192, [8192, 5000], 137, True)
    q, k, v = inp.q.cuda(), inp.k.cuda(), inp.v.cuda()
    lens = inp.kv_lengths.cuda()
    mask_d = chunk_mask(2, 2, 8192, 138).cuda()
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    ws = make_ws(inp, "tc")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        fd.decode_masked(q, k, v, lens, mask_d, n_q=2, causal=True, scale=inp.scale, out=out,
                         kernel=fd.FD_KERNEL_TC, workspace=ws, stream=s)
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        fd.decode_masked(q, k, v, lens, mask_d, n_q=2, causal=True, scale=inp.scale, out=out,
                         kernel=fd.FD_KERNEL_TC, workspace=ws, stream=s)
    for seed, new_lens in ((139, [8192, 5000]), (140, [3001, 7777])):
        mask = chunk_mask(2, 2, 8192, seed, keep=0.2)
        mask_d.copy_(mask)
        lens.copy_(torch.tensor(new_lens, dtype=torch.int32))
        graph.replay()
        torch.cuda.synchronize()
        ref = torch.from_numpy(oracle.masked(inp.q, inp.k, inp.v,
                                             torch.tensor(new_lens, dtype=torch.int32), mask, 2,
                                             True, inp.scale))
        compare(out, ref, torch.float32, "graph replay %d" % seed)
    assert ws.device_status() == 0
    ws.close()
