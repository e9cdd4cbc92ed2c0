"""GPU parity of the fused-append call (fd_decode_append) against the fp64
oracle: the output, the cache contents after the step (bit for bit) and the
updated lengths, for both kernels, windows of 1-6 new rows, new rows that
straddle tile boundaries, ragged and empty sequences, rows past the
capacity, split counts, a CUDA-graph decode loop and the full-size ragged
workload."""
import numpy as np
import pytest
import torch

import oracle
from decode_attention_preallocated_gb300 import build as fdbuild
from decode_attention_preallocated_gb300 import fd
from decode_attention_preallocated_gb300 import workloads as W
from parity_util import compare

pytestmark = pytest.mark.gpu

KERNELS = [fd.FD_KERNEL_SIMT, fd.FD_KERNEL_TC]


@pytest.fixture(scope="module", autouse=True)
def _built():
    fdbuild.build()
    fd.lib()


def make(B, n, Hq, Hkv, d, cap, lens, causal, seed, tail="randn"):
    inp = W.dense_inputs(B, n, Hq, Hkv, d, cap, lens, seed, causal, tail=tail)
    g = torch.Generator().manual_seed(seed + 1)
    kn = W.randn_bf16((B, n, Hkv, d), g, "cpu")
    vn = W.randn_bf16((B, n, Hkv, d), g, "cpu")
    return inp, kn, vn


def bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def run_step(inp, kn, vn, out_dtype, kernel, update=True, num_ctas=0, ws=None):
    """One fused step on the GPU; returns (out, k, v, lengths, status)."""
    q, k, v = inp.q.cuda(), inp.k.cuda(), inp.v.cuda()
    lens = inp.kv_lengths.cuda()
    own = ws is None
    if own:
        B, n, Hq, d = inp.q.shape
        ws = fd.Workspace(B * inp.k.shape[1], min(64, (Hq // inp.k.shape[1]) * n), 256,
                          max(2048, num_ctas))
    out = fd.decode_append(q, k, v, kn.cuda(), vn.cuda(), lens, causal=inp.causal,
                           scale=inp.scale, update_lengths=update, out_dtype=out_dtype,
                           kernel=kernel, num_ctas=num_ctas, workspace=ws)
    torch.cuda.synchronize()
    st = ws.diagnostics()
    assert not st[0] & fd.FD_DEV_INTERNAL, "internal error: site %d tile %d piece %d" % tuple(st[1:4])
    if own:
        ws.close()
    return out, k, v, lens, st[0]


def check_step(inp, kn, vn, out_dtype, kernel, update=True, num_ctas=0):
    ref, ka, va, after = oracle.append(inp.q, inp.k, inp.v, kn, vn, inp.kv_lengths,
                                       inp.causal, inp.scale)
    out, k, v, lens, status = run_step(inp, kn, vn, out_dtype, kernel, update, num_ctas)
    compare(out, torch.from_numpy(ref), out_dtype, "append")
    assert np.array_equal(bits(k), ka), "k cache after the step"
    assert np.array_equal(bits(v), va), "v cache after the step"
    want = after if update else inp.kv_lengths.numpy()
    assert lens.cpu().numpy().tolist() == list(want), (lens.cpu().tolist(), list(want))
    return status


SMALL = {
    # name: (B, n_new, Hq, Hkv, d, cap, lengths before, causal)
    "mtp_d256": (1, 4, 16, 4, 256, 1201, [995], True),
    "ragged_d256": (4, 6, 16, 4, 256, 700, [0, 60, 330, 690], True),
    "tile_edge_d128": (2, 4, 8, 2, 128, 400, [126, 252], True),
    "decode1_d128": (3, 1, 8, 2, 128, 600, [517, 1, 599], False),
    "rows64_d128": (2, 2, 32, 1, 128, 300, [200, 77], True),
    "noncausal_d256": (2, 3, 8, 2, 256, 500, [129, 300], False),
}


@pytest.mark.parametrize("case", sorted(SMALL))
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("kernel", KERNELS)
def test_append_small(case, out_dtype, kernel):
    B, n, Hq, Hkv, d, cap, lens, causal = SMALL[case]
    inp, kn, vn = make(B, n, Hq, Hkv, d, cap, lens, causal, 60)
    check_step(inp, kn, vn, out_dtype, kernel)


@pytest.mark.parametrize("kernel", KERNELS)
def test_append_without_length_update(kernel):
    inp, kn, vn = make(2, 3, 8, 2, 128, 300, [100, 250], True, 61)
    check_step(inp, kn, vn, torch.float32, kernel, update=False)


@pytest.mark.parametrize("kernel", KERNELS)
def test_append_past_the_capacity_is_clamped_and_flagged(kernel):
    inp, kn, vn = make(2, 4, 8, 2, 128, 300, [298, 50], True, 62)
    status = check_step(inp, kn, vn, torch.float32, kernel)
    assert status & fd.FD_DEV_BAD_LENGTH


@pytest.mark.parametrize("kernel,ctas", [(fd.FD_KERNEL_TC, 1), (fd.FD_KERNEL_TC, 7),
                                         (fd.FD_KERNEL_TC, 100), (fd.FD_KERNEL_SIMT, 1),
                                         (fd.FD_KERNEL_SIMT, 300)])
def test_append_split_counts(kernel, ctas):
    inp, kn, vn = make(3, 4, 16, 4, 256, 900, [896, 27, 450], True, 63)
    check_step(inp, kn, vn, torch.float32, kernel, num_ctas=ctas)


def test_append_tensor_core_rejects_more_blocks_than_resident():
    inp, kn, vn = make(1, 2, 8, 2, 128, 300, [100], True, 64)
    with pytest.raises(fd.FdError):
        run_step(inp, kn, vn, torch.float32, fd.FD_KERNEL_TC, num_ctas=5000)


@pytest.mark.parametrize("kernel", KERNELS)
def test_append_graph_decode_loop(kernel):
    # one captured step, replayed: each replay appends the next token (new
    # q / k_new / v_new copied into the step's input buffers first) and
    # advances the lengths on the device
    B, Hq, Hkv, d, cap = 2, 16, 4, 256, 700
    inp, _, _ = make(B, 1, Hq, Hkv, d, cap, [300, 41], True, 65)
    g = torch.Generator().manual_seed(66)
    steps = [(W.randn_bf16((B, 1, Hq, d), g, "cpu"), W.randn_bf16((B, 1, Hkv, d), g, "cpu"),
              W.randn_bf16((B, 1, Hkv, d), g, "cpu")) for _ in range(5)]
    q = torch.empty_like(inp.q).cuda()
    kn = torch.empty((B, 1, Hkv, d), dtype=torch.bfloat16, device="cuda")
    vn = torch.empty_like(kn)
    k, v, lens = inp.k.cuda(), inp.v.cuda(), inp.kv_lengths.cuda()
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    ws = fd.Workspace(B * Hkv, Hq // Hkv, 256, 2048)

    def call():
        fd.decode_append(q, k, v, kn, vn, lens, causal=True, scale=inp.scale, out=out,
                         kernel=kernel, workspace=ws)

    s = torch.cuda.Stream()
    # warm-up call on a scratch copy so the real cache sees only the replays
    q.copy_(steps[0][0]); kn.copy_(steps[0][1]); vn.copy_(steps[0][2])
    k0, v0, l0 = k.clone(), v.clone(), lens.clone()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    k.copy_(k0); v.copy_(v0); lens.copy_(l0)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        call()
    # the capture ran nothing: the cache and lengths are still the originals
    kh, vh, lh = inp.k.clone(), inp.v.clone(), inp.kv_lengths.clone()
    for qs, kns, vns in steps:
        q.copy_(qs); kn.copy_(kns); vn.copy_(vns)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        ref, ka, va, after = oracle.append(qs, kh, vh, kns, vns, lh, True, inp.scale)
        compare(out, torch.from_numpy(ref), torch.float32, "graph step")
        kh = torch.from_numpy(ka.view(np.int16)).view(torch.bfloat16)
        vh = torch.from_numpy(va.view(np.int16)).view(torch.bfloat16)
        lh = torch.from_numpy(after)
        assert lens.cpu().tolist() == after.tolist()
    assert np.array_equal(bits(k), bits(kh)) and np.array_equal(bits(v), bits(vh))
    ws.close()


@pytest.mark.parametrize("kernel", KERNELS)
def test_append_full_size_ragged(kernel):
    # the ragged workload as a fused step: 6 new rows per sequence appended to
    # its first L - 6 positions
    inp = W.workload("ragged", seed=1)
    g = torch.Generator().manual_seed(67)
    B, n, Hq, d = inp.q.shape
    Hkv = inp.k.shape[1]
    kn = W.randn_bf16((B, n, Hkv, d), g, "cpu")
    vn = W.randn_bf16((B, n, Hkv, d), g, "cpu")
    inp.kv_lengths = inp.kv_lengths - n
    check_step(inp, kn, vn, torch.bfloat16, kernel)
