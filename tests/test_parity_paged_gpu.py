"""GPU parity of the paged-cache calls (fd_decode_paged) against the fp64
oracle: page sizes from 1 to 256 (powers of two and not), both pool layouts,
causal windows, ragged lengths, split counts, bad table entries, poisoned
free rows, int8 pools, graph replay with new lengths and tables, and the
full-size paged workloads."""
import pytest
import torch

from decode_attention_preallocated_gb300 import build as fdbuild
from decode_attention_preallocated_gb300 import fd
from decode_attention_preallocated_gb300 import workloads as W
from parity_util import compare, run_gpu, run_oracle, to_dev

pytestmark = pytest.mark.gpu

KERNELS = [fd.FD_KERNEL_SIMT, fd.FD_KERNEL_TC]


@pytest.fixture(scope="module", autouse=True)
def _built():
    fdbuild.build()
    fd.lib()


def check(inp, out_dtype=torch.bfloat16, num_ctas=0, kernel=fd.FD_KERNEL_AUTO, ref=None):
    if ref is None:
        ref = run_oracle(inp)
    got = run_gpu(to_dev(inp), out_dtype, num_ctas, kernel)
    torch.cuda.synchronize()
    return compare(got, ref, out_dtype, inp.name or "paged"), got


SMALL = {
    # name: (B, n_q, Hq, Hkv, d, page_size, max_pages, lengths, causal)
    "d128_ps64": (3, 1, 8, 2, 128, 64, 12, [700, 65, 1], False),
    "d256_ps16_mtp": (2, 4, 16, 4, 256, 16, 40, [640, 333], True),
    "d256_ps128_ragged6": (4, 6, 16, 4, 256, 128, 6, [768, 1, 129, 500], True),
    "d128_ps1": (1, 2, 8, 2, 128, 1, 300, [300], True),
    "d128_ps100": (2, 3, 12, 3, 128, 100, 7, [650, 99], True),
    "d256_ps256": (2, 2, 8, 1, 256, 256, 3, [768, 257], True),
    "rows64_ps32": (2, 2, 32, 1, 128, 32, 10, [300, 77], True),
}


@pytest.mark.parametrize("case", sorted(SMALL))
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("kernel", KERNELS)
def test_paged_small(case, out_dtype, kernel):
    B, n_q, Hq, Hkv, d, ps, mp, lens, causal = SMALL[case]
    inp = W.paged_inputs(B, n_q, Hq, Hkv, d, ps, mp, lens, 31, causal, name=case)
    check(inp, out_dtype, kernel=kernel)


@pytest.mark.parametrize("kernel", KERNELS)
def test_paged_token_major_pool(kernel):
    inp = W.paged_inputs(2, 3, 8, 2, 128, 48, 9, [400, 47], 32, True, layout="bthd")
    assert inp.k.stride(2) == 2 * 128
    check(inp, torch.float32, kernel=kernel)


@pytest.mark.parametrize("kernel", KERNELS)
def test_paged_free_rows_are_never_read(kernel):
    # NaN in every pool row that holds no position below its length
    clean = W.paged_inputs(3, 4, 16, 4, 256, 64, 8, [500, 64, 3], 33, True)
    poisoned = W.paged_inputs(3, 4, 16, 4, 256, 64, 8, [500, 64, 3], 33, True, tail="nan")
    ref = run_oracle(clean)
    (_, _, _), got = check(poisoned, torch.float32, kernel=kernel, ref=ref)
    assert torch.isfinite(got).all()


@pytest.mark.parametrize("ctas", [1, 3, 19, 300])
def test_paged_tensor_core_splits(ctas):
    inp = W.paged_inputs(3, 6, 16, 4, 256, 16, 60, [960, 17, 511], 34, True)
    ref = run_oracle(inp)
    check(inp, torch.float32, kernel=fd.FD_KERNEL_TC, num_ctas=ctas, ref=ref)
    check(inp, torch.bfloat16, kernel=fd.FD_KERNEL_TC, num_ctas=ctas, ref=ref)


@pytest.mark.parametrize("kernel", KERNELS)
def test_paged_bad_table_entry_is_skipped_and_flagged(kernel):
    inp = W.paged_inputs(2, 2, 8, 2, 128, 32, 10, [300, 200], 35, True)
    inp.block_table = inp.block_table.clone()
    inp.block_table[0, 3] = -1                          # positions 96..127 of sequence 0
    inp.block_table[1, 2] = inp.k.shape[0] + 11         # positions 64..95 of sequence 1
    inp.block_table[1, 9] = -5                          # past the length: never read
    ref = run_oracle(inp)
    dev = to_dev(inp)
    ws = fd.Workspace(8, 64, 256, 1024)
    got = run_gpu(dev, torch.float32, kernel=kernel, workspace=ws)
    torch.cuda.synchronize()
    assert ws.device_status() & fd.FD_DEV_BAD_INDEX
    compare(got, ref, torch.float32, "bad pages")
    ws.close()


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("causal,n_q", [(False, 1), (True, 4)])
def test_paged_int8(kernel, causal, n_q):
    inp = W.paged_inputs(3, n_q, 32, 8, 128, 64, 10, [640, 200, 1], 36, causal, int8=True)
    check(inp, torch.bfloat16, kernel=kernel)
    check(inp, torch.float32, kernel=kernel)


@pytest.mark.parametrize("kernel", KERNELS)
def test_paged_int8_poisoned_free_scales(kernel):
    inp = W.paged_inputs(2, 4, 32, 4, 128, 16, 40, [600, 33], 37, True, int8=True, tail="nan")
    check(inp, torch.float32, kernel=kernel)


@pytest.mark.parametrize("ctas", [1, 19, 300])
def test_paged_int8_tensor_core_splits(ctas):
    inp = W.paged_inputs(3, 4, 32, 4, 128, 128, 12, [1500, 611, 129], 38, True, int8=True)
    check(inp, torch.float32, kernel=fd.FD_KERNEL_TC, num_ctas=ctas)


@pytest.mark.parametrize("ps", [16, 64, 100, 256])
def test_paged_int8_head_dim_256_tensor_core(ps):
    # head_dim 256 int8 pools: page runs of 16 / 64 / 256 positions, and a
    # page size (100) whose tiles are gathered row by row
    inp = W.paged_inputs(3, 4, 16, 4, 256, ps, 2000 // ps + 1, [1500, 611, 129], 40, True,
                         int8=True, tail="nan")
    check(inp, torch.float32, kernel=fd.FD_KERNEL_TC)
    check(inp, torch.bfloat16, kernel=fd.FD_KERNEL_TC)


def test_paged_layout_that_no_row_view_covers_falls_back():
    # pool rows padded to 136 elements and a page stride that is not a
    # multiple of the row stride: the tensor-core kernel declines, AUTO takes
    # the CUDA-core one
    inp = W.paged_inputs(2, 1, 8, 2, 128, 16, 6, [90, 40], 39, False)
    P, H, ps, d = inp.k.shape
    buf_k = torch.zeros(P * (H * ps * 136 + 8), dtype=torch.bfloat16)
    buf_v = torch.zeros_like(buf_k)
    strides = (H * ps * 136 + 8, ps * 136, 136, 1)
    k = torch.as_strided(buf_k, (P, H, ps, d), strides)
    v = torch.as_strided(buf_v, (P, H, ps, d), strides)
    k.copy_(inp.k)
    v.copy_(inp.v)
    ref = run_oracle(inp)
    dev = to_dev(inp)
    dev.k = torch.as_strided(buf_k.cuda(), (P, H, ps, d), strides)
    dev.v = torch.as_strided(buf_v.cuda(), (P, H, ps, d), strides)
    with pytest.raises(fd.FdError):
        run_gpu(dev, torch.float32, kernel=fd.FD_KERNEL_TC)
    compare(run_gpu(dev, torch.float32), ref, torch.float32, "paged strided pool")


@pytest.mark.parametrize("kernel", KERNELS)
def test_paged_graph_replay_with_new_lengths_and_tables(kernel):
    inp = W.paged_inputs(2, 4, 16, 4, 256, 32, 20, [640, 640], 40, True, spare_pages=8)
    dev = to_dev(inp)
    ws = fd.Workspace(16, 64, 256, 1024)
    out = torch.empty(dev.q.shape, dtype=torch.float32, device="cuda")

    def call():
        fd.decode_paged(dev.q, dev.k, dev.v, dev.block_table, dev.kv_lengths, n_q=4,
                        causal=True, scale=inp.scale, out=out, kernel=kernel, workspace=ws)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        call()
    gen = torch.Generator().manual_seed(41)
    P = inp.k.shape[0]
    for lens in ([640, 640], [17, 639], [513, 4], [0, 100]):
        table = torch.randperm(P, generator=gen)[:40].view(2, 20).to(torch.int32)
        dev.block_table.copy_(table)
        dev.kv_lengths.copy_(torch.tensor(lens, dtype=torch.int32))
        graph.replay()
        torch.cuda.synchronize()
        inp.block_table = table
        inp.kv_lengths = torch.tensor(lens, dtype=torch.int32)
        compare(out, run_oracle(inp), torch.float32, "paged graph replay %s" % lens)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("name", W.PAGED_WORKLOADS)
def test_paged_workload_full_size(kernel, name):
    # the full-size paged workloads, generated on the GPU; every output row
    # is checked against the oracle on the same bits
    inp = W.workload(name, seed=1, device="cuda")
    got = run_gpu(inp, torch.bfloat16, kernel=kernel)
    torch.cuda.synchronize()
    cpu = W.DecodeInputs(q=inp.q.cpu(), k=inp.k.cpu(), v=inp.v.cpu(),
                         kv_lengths=inp.kv_lengths.cpu(), n_q=inp.n_q, causal=inp.causal,
                         scale=inp.scale,
                         k_scale=None if inp.k_scale is None else inp.k_scale.cpu(),
                         v_scale=None if inp.v_scale is None else inp.v_scale.cpu(),
                         block_table=inp.block_table.cpu(), page_size=inp.page_size)
    compare(got, run_oracle(cpu), torch.bfloat16, name)
