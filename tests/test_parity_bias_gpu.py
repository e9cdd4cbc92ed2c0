"""GPU parity of the biased index gather (fd_decode_gather_bias) against the
fp64 oracle, for both kernels: seeded N(0, 2) biases with -inf entries and a
row that is -inf throughout, large biases that decide the softmax, head_dim
128 and 256, a token-major cache, and the full-size gather workload."""
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


def seeded_bias(idx, seed, spread=2.0):
    g = torch.Generator().manual_seed(seed)
    bias = torch.randn(idx.shape, generator=g) * spread
    drop = torch.rand(idx.shape, generator=g) < 0.1
    bias[drop] = -float("inf")
    bias[0, -1, :] = -float("inf")          # a row with nothing left: zeros
    return bias


def run(inp, bias, out_dtype, kernel, k=None, v=None, num_ctas=0):
    ws = fd.Workspace(inp.q.shape[0] * inp.q.shape[1] * inp.k.shape[1], 64, 256, 2048)
    out = fd.decode_gather(inp.q.cuda(), (inp.k if k is None else k).cuda(),
                           (inp.v if v is None else v).cuda(), inp.idx.cuda(),
                           scale=inp.scale, out_dtype=out_dtype, kernel=kernel,
                           num_ctas=num_ctas, workspace=ws, bias=bias.cuda())
    torch.cuda.synchronize()
    st = ws.diagnostics()
    assert not st[0] & fd.FD_DEV_INTERNAL
    assert not st[0] & fd.FD_DEV_BAD_INDEX     # -inf entries are not bad cells
    ws.close()
    return out


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("d", [128, 256])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_biased_gather(kernel, d, out_dtype):
    inp = W.gather_inputs(2, 3, 32, 4, d, 3000, 700, 64, seed=41)
    bias = seeded_bias(inp.idx, 42)
    ref = torch.from_numpy(oracle.gather(inp.q, inp.k, inp.v, inp.idx, inp.scale, bias=bias))
    got = run(inp, bias, out_dtype, kernel)
    compare(got, ref, out_dtype, "biased gather")
    assert torch.count_nonzero(got[0, -1].cpu()) == 0


@pytest.mark.parametrize("kernel", KERNELS)
def test_large_biases_decide_the_softmax(kernel):
    inp = W.gather_inputs(1, 2, 16, 2, 128, 2000, 300, 16, seed=43)
    bias = seeded_bias(inp.idx, 44, spread=30.0)
    ref = torch.from_numpy(oracle.gather(inp.q, inp.k, inp.v, inp.idx, inp.scale, bias=bias))
    for od in (torch.float32, torch.bfloat16):
        compare(run(inp, bias, od, kernel), ref, od, "large biases")


@pytest.mark.parametrize("ctas", [1, 5, 64])
def test_biased_gather_tensor_core_splits_token_major(ctas):
    inp = W.gather_inputs(2, 2, 16, 4, 256, 4000, 1500, 128, seed=45)
    bias = seeded_bias(inp.idx, 46)
    ref = torch.from_numpy(oracle.gather(inp.q, inp.k, inp.v, inp.idx, inp.scale, bias=bias))
    k = inp.k.transpose(1, 2).contiguous().transpose(1, 2)
    v = inp.v.transpose(1, 2).contiguous().transpose(1, 2)
    got = run(inp, bias, torch.float32, fd.FD_KERNEL_TC, k=k, v=v, num_ctas=ctas)
    compare(got, ref, torch.float32, "biased gather token-major")


@pytest.mark.parametrize("kernel", KERNELS)
def test_biased_gather_workload_full_size(kernel):
    inp = W.workload("gather", seed=1)
    bias = seeded_bias(inp.idx, 47)
    bias[0, -1, :] = 0.0
    ref = torch.from_numpy(oracle.gather(inp.q, inp.k, inp.v, inp.idx, inp.scale, bias=bias))
    compare(run(inp, bias, torch.bfloat16, kernel), ref, torch.bfloat16, "gather workload, bias")
