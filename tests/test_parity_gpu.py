"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
the same seeded inputs, element by element, for every mode and the edge
cases.  Sizes span several tiles and a ragged tail; the named workloads also
run at full size."""
import math

import pytest
import torch

from decode_attention_preallocated_gb300 import build as fdbuild
from decode_attention_preallocated_gb300 import fd
from decode_attention_preallocated_gb300 import workloads as W
from golden_cases import fixture_names, load as load_fixture
from parity_util import TOL, compare, run_gpu, run_oracle, to_dev

pytestmark = pytest.mark.gpu

KERNELS = [fd.FD_KERNEL_SIMT]
DENSE_KERNELS = [fd.FD_KERNEL_SIMT, fd.FD_KERNEL_TC]
INT8_KERNELS = [fd.FD_KERNEL_SIMT, fd.FD_KERNEL_TC]   # tensor cores: <= 32 rows a launch
GATHER_KERNELS = [fd.FD_KERNEL_SIMT, fd.FD_KERNEL_TC]


@pytest.fixture(scope="module", autouse=True)
def _built():
    fdbuild.build()
    fd.lib()


def check(inp_cpu, out_dtype=torch.bfloat16, num_ctas=0, kernel=fd.FD_KERNEL_AUTO,
          ref=None, what=""):
    if ref is None:
        ref = run_oracle(inp_cpu)
    dev = to_dev(inp_cpu)
    got = run_gpu(dev, out_dtype, num_ctas, kernel)
    torch.cuda.synchronize()
    return compare(got, ref, out_dtype, what or inp_cpu.name), got


# --------------------------------------------------------------- fixtures
@pytest.mark.parametrize("name", fixture_names())
@pytest.mark.parametrize("d", [128, 256])
@pytest.mark.parametrize("kernel", DENSE_KERNELS)
def test_golden_fixture_on_gpu(name, d, kernel):
    fx = load_fixture(name, pad_d=d)
    dev = lambda t: None if t is None else t.cuda()
    for out_dtype in (torch.float32, torch.bfloat16):
        if fx["mode"] == "gather":
            got = fd.decode_gather(dev(fx["q"]), dev(fx["k"]), dev(fx["v"]), dev(fx["idx"]),
                                   scale=fx["scale"], out_dtype=out_dtype, kernel=kernel)
        elif fx.get("int8"):
            got = fd.decode_int8(dev(fx["q"]), dev(fx["k"]), dev(fx["v"]),
                                 dev(fx["k_scale"]), dev(fx["v_scale"]),
                                 dev(fx["kv_lengths"]), n_q=fx["n_q"], causal=fx["causal"],
                                 scale=fx["scale"], out_dtype=out_dtype, kernel=kernel)
        else:
            got = fd.decode(dev(fx["q"]), dev(fx["k"]), dev(fx["v"]), dev(fx["kv_lengths"]),
                            n_q=fx["n_q"], causal=fx["causal"], scale=fx["scale"],
                            out_dtype=out_dtype, kernel=kernel)
        compare(got, fx["expected"], out_dtype, name)


# ---------------------------------------------------- reduced-size workloads
SMALL = {
    # name: (B, n_q, Hq, Hkv, d, cap, lengths, causal)
    "dense_d128": (1, 1, 8, 2, 128, 600, [517], False),
    "mtp_d256": (1, 4, 16, 4, 256, 1201, [999], True),
    "ragged_d256": (4, 6, 16, 4, 256, 700, [1, 65, 333, 700], True),
    "ragged_d128": (3, 3, 12, 3, 128, 450, [450, 7, 129], True),
    "mqa_rows64": (2, 2, 32, 1, 128, 300, [300, 77], True),
    "mha_g1": (2, 5, 3, 3, 256, 260, [2, 259], True),
}


@pytest.mark.parametrize("case", sorted(SMALL))
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("kernel", DENSE_KERNELS)
def test_dense_small(case, out_dtype, kernel):
    B, n_q, Hq, Hkv, d, cap, lens, causal = SMALL[case]
    inp = W.dense_inputs(B, n_q, Hq, Hkv, d, cap, lens, 11, causal, name=case)
    check(inp, out_dtype, kernel=kernel)


@pytest.mark.parametrize("kernel", DENSE_KERNELS)
@pytest.mark.parametrize("num_ctas", [1, 2, 3, 7, 19, 64, 300, 1000])
def test_split_count_does_not_change_result(kernel, num_ctas):
    inp = W.dense_inputs(3, 4, 16, 4, 256, 900, [900, 31, 450], 12, True)
    ref = run_oracle(inp)
    check(inp, torch.float32, num_ctas=num_ctas, kernel=kernel, ref=ref)


@pytest.mark.parametrize("kernel", DENSE_KERNELS)
@pytest.mark.parametrize("num_ctas", [32, 48, 100, 152])
@pytest.mark.parametrize("n_q", [1, 4, 6])
def test_short_head_dim_256_launch_merges(kernel, num_ctas, n_q):
    # one 3000-position sequence at head_dim 256 over 4 kv heads: a short
    # launch, whose split segments the tensor-core kernel merges in shares;
    # the grid sets the pieces per segment (about 8 to 30) and with the rows
    # (4, 16 or 24) the threads that share one output unit's pieces (1 to
    # about 30)
    inp = W.dense_inputs(1, n_q, 16, 4, 256, 3000, [3000], 17, True)
    check(inp, torch.float32, num_ctas=num_ctas, kernel=kernel)


@pytest.mark.parametrize("kernel", DENSE_KERNELS)
def test_capacity_beyond_length_is_never_read(kernel):
    # NaN in every cache row past the length, capacities from L to 4L
    L = 700
    base = W.dense_inputs(2, 4, 16, 4, 256, L, [L, L], 13, True)
    ref = run_oracle(base)
    for cap in (L, L + 1, 2 * L + 3, 4 * L):
        inp = W.dense_inputs(2, 4, 16, 4, 256, cap, [L, L], 13, True, tail="nan")
        inp.q.copy_(base.q)
        inp.k[:, :, :L] = base.k
        inp.v[:, :, :L] = base.v
        (mx, _, _), got = check(inp, torch.float32, kernel=kernel, ref=ref)


@pytest.mark.parametrize("kernel", DENSE_KERNELS)
def test_token_major_cache_layout(kernel):
    inp = W.dense_inputs(2, 3, 8, 2, 128, 333, [333, 100], 14, True, layout="bthd")
    assert inp.k.stride(2) == 2 * 128
    check(inp, torch.float32, kernel=kernel)


@pytest.mark.parametrize("kernel", DENSE_KERNELS)
def test_empty_windows_give_zero(kernel):
    # L = 0, and causal rows whose window would start before position 0
    inp = W.dense_inputs(3, 6, 8, 2, 128, 64, [0, 3, 64], 15, True)
    (_, _, _), got = check(inp, torch.float32, kernel=kernel)
    g = got.cpu()
    assert torch.count_nonzero(g[0]) == 0
    assert torch.count_nonzero(g[1, :3]) == 0


@pytest.mark.parametrize("kernel", DENSE_KERNELS)
def test_bad_lengths_are_clamped_and_flagged(kernel):
    inp = W.dense_inputs(2, 1, 8, 2, 128, 100, [100, 100], 16, False)
    dev = to_dev(inp)
    dev.kv_lengths = torch.tensor([-5, 1000], dtype=torch.int32, device="cuda")
    ws = fd.Workspace(8, 16, 256, 1024)
    got = run_gpu(dev, torch.float32, kernel=kernel, workspace=ws)
    torch.cuda.synchronize()
    assert ws.device_status() & fd.FD_DEV_BAD_LENGTH
    inp.kv_lengths = torch.tensor([0, 100], dtype=torch.int32)
    compare(got, run_oracle(inp), torch.float32, "clamped lengths")
    ws.reset()
    assert ws.device_status() == 0


@pytest.mark.parametrize("kernel", DENSE_KERNELS)
def test_peaky_scores(kernel):
    # q scaled x8: outputs are O(1), so absolute tolerances bite
    inp = W.dense_inputs(2, 2, 8, 2, 256, 400, [400, 250], 17, True, q_mult=8.0)
    ref = run_oracle(inp)
    assert float(ref.abs().max()) > 1.0
    check(inp, torch.float32, kernel=kernel, ref=ref)
    check(inp, torch.bfloat16, kernel=kernel, ref=ref)


@pytest.mark.parametrize("kernel", DENSE_KERNELS)
def test_rollback_by_length(kernel):
    inp = W.dense_inputs(1, 4, 16, 4, 256, 800, [703], 18, True)
    dev = to_dev(inp)
    a = run_gpu(dev, torch.float32, kernel=kernel)
    dev.kv_lengths.fill_(700)               # reject three drafts
    b = run_gpu(dev, torch.float32, kernel=kernel)
    fresh = W.dense_inputs(1, 4, 16, 4, 256, 800, [700], 18, True)
    compare(b, run_oracle(fresh), torch.float32, "rolled back")
    compare(a, run_oracle(inp), torch.float32, "before rollback")


@pytest.mark.parametrize("kernel", DENSE_KERNELS)
def test_causal_row_ignores_later_drafts(kernel):
    n_q, L = 6, 500
    a = W.dense_inputs(1, n_q, 16, 4, 256, 512, [L], 19, True)
    b = W.dense_inputs(1, n_q, 16, 4, 256, 512, [L], 19, True)
    b.k[:, :, L - 3:L] = 5.0
    b.v[:, :, L - 3:L] = -9.0
    ga = run_gpu(to_dev(a), torch.float32, kernel=kernel).cpu()
    gb = run_gpu(to_dev(b), torch.float32, kernel=kernel).cpu()
    # rows 0..2 see positions <= L-4 only
    assert torch.equal(ga[0, :3], gb[0, :3])
    assert not torch.equal(ga[0, 3:], gb[0, 3:])


# ------------------------------------------------------------------ gather
@pytest.mark.parametrize("kernel", GATHER_KERNELS)
@pytest.mark.parametrize("n_q", [1, 3])
def test_gather_small(kernel, n_q):
    inp = W.gather_inputs(2, n_q, 32, 4, 128, 3000, 200, 16, 20)
    inp.idx[0, 0, 5] = -1
    inp.idx[1, n_q - 1, 7] = -3
    check(inp, torch.float32, kernel=kernel)
    check(inp, torch.bfloat16, kernel=kernel)


@pytest.mark.parametrize("kernel", GATHER_KERNELS)
def test_gather_prefix_equals_dense(kernel):
    L = 333
    inp = W.dense_inputs(1, 1, 8, 2, 128, 400, [L], 21, False)
    dev = to_dev(inp)
    dense = run_gpu(dev, torch.float32, kernel=kernel)
    idx = torch.arange(L, dtype=torch.int32, device="cuda").view(1, 1, L)
    g = fd.decode_gather(dev.q, dev.k, dev.v, idx, scale=inp.scale,
                         out_dtype=torch.float32, kernel=kernel)
    # the same cells in other tiles: rounding-level differences only (P is
    # carried to ~2^-17 on the tensor cores, fp32 on the CUDA cores)
    tol = 2e-6 if kernel == fd.FD_KERNEL_SIMT else 1e-4
    torch.testing.assert_close(g, dense, rtol=0, atol=tol)
    perm = idx[:, :, torch.randperm(L, device="cuda")].contiguous()
    g2 = fd.decode_gather(dev.q, dev.k, dev.v, perm, scale=inp.scale,
                          out_dtype=torch.float32, kernel=kernel)
    torch.testing.assert_close(g2, dense, rtol=0, atol=tol)


@pytest.mark.parametrize("kernel", GATHER_KERNELS)
def test_gather_out_of_range_index_is_skipped_and_flagged(kernel):
    inp = W.gather_inputs(1, 1, 8, 2, 128, 500, 64, 4, 22)
    dev = to_dev(inp)
    dev.idx[0, 0, 3] = 500
    dev.idx[0, 0, 9] = 1 << 30
    ws = fd.Workspace(8, 16, 256, 1024)
    got = fd.decode_gather(dev.q, dev.k, dev.v, dev.idx, scale=inp.scale,
                           out_dtype=torch.float32, kernel=kernel, workspace=ws)
    torch.cuda.synchronize()
    assert ws.device_status() & fd.FD_DEV_BAD_INDEX
    inp.idx = dev.idx.cpu()
    compare(got, run_oracle(inp), torch.float32, "gather skip")


@pytest.mark.parametrize("kernel", GATHER_KERNELS)
def test_gather_empty_list(kernel):
    inp = W.gather_inputs(1, 2, 8, 2, 128, 100, 8, 2, 23)
    dev = to_dev(inp)
    idx = torch.full((1, 2, 8), -1, dtype=torch.int32, device="cuda")
    got = fd.decode_gather(dev.q, dev.k, dev.v, idx, out_dtype=torch.float32, kernel=kernel)
    assert torch.count_nonzero(got) == 0
    idx0 = torch.empty((1, 2, 0), dtype=torch.int32, device="cuda")
    got = fd.decode_gather(dev.q, dev.k, dev.v, idx0, out_dtype=torch.float32, kernel=kernel)
    assert torch.count_nonzero(got) == 0


@pytest.mark.parametrize("ctas", [1, 5, 64, 300])
@pytest.mark.parametrize("d", [128, 256])
def test_gather_tensor_core_splits_token_major(ctas, d):
    # lists of 700 cells over a token-major cache, many split pieces
    inp = W.gather_inputs(2, 2, 16, 4, d, 4000, 700, 64, 28)
    inp.idx[1, 1, 33] = -1
    tm = to_dev(inp)
    k = tm.k.transpose(1, 2).contiguous().transpose(1, 2)   # [B, cap, Hkv, d] storage
    v = tm.v.transpose(1, 2).contiguous().transpose(1, 2)
    for od in (torch.float32, torch.bfloat16):
        got = fd.decode_gather(tm.q, k, v, tm.idx, scale=inp.scale, out_dtype=od,
                               kernel=fd.FD_KERNEL_TC, num_ctas=ctas)
        compare(got, run_oracle(inp), od, "gather tc token-major")


@pytest.mark.parametrize("d", [128, 256])
@pytest.mark.parametrize("g,idx_len", [(8, 2048), (4, 300), (16, 129), (32, 1000), (64, 640)])
def test_gather_tensor_core_cluster_merges(d, g, idx_len):
    # automatic grid: lists of 2-16 tiles whose clusters all fit the device
    # merge through distributed shared memory (129 entries: a one-entry last
    # tile; 64 rows: the widest instantiation); the same inputs on an
    # explicit grid take the global merge.  Both against the oracle, with
    # padding and an out-of-range cell in the lists.
    B, n_q, Hkv = (1, 1, 4) if g >= 32 else (2, 2, 2)
    inp = W.gather_inputs(B, n_q, g * Hkv, Hkv, d, 5000, idx_len, min(64, idx_len), 43)
    inp.idx[0, 0, 3] = -1
    inp.idx[-1, -1, idx_len // 2] = 5000
    ref = run_oracle(inp)
    for ctas in (0, 37):
        for od in (torch.float32, torch.bfloat16):
            check(inp, od, kernel=fd.FD_KERNEL_TC, num_ctas=ctas, ref=ref,
                  what="gather d%d g%d len%d ctas%d" % (d, g, idx_len, ctas))


@pytest.mark.parametrize("kernel", GATHER_KERNELS)
@pytest.mark.parametrize("d,g,ctas", [(128, 8, 0), (128, 16, 7), (256, 4, 0), (256, 32, 300)])
def test_gather_int8(kernel, d, g, ctas):
    # int8 caches with per-cell scales: padding, an out-of-range cell, lists
    # longer than a tile, 8 / 16 / 4 / 32 query heads per kv head
    inp = W.gather_inputs(2, 2, 4 * g, 4, d, 3000, 300, 32, 41, int8=True)
    inp.idx[0, 0, 5] = -1
    inp.idx[1, 1, 9] = 3000
    check(inp, torch.float32, kernel=kernel, num_ctas=ctas)
    check(inp, torch.bfloat16, kernel=kernel, num_ctas=ctas)


@pytest.mark.parametrize("kernel", GATHER_KERNELS)
def test_gather_int8_workload_shape(kernel):
    # the gather workload's shape (2048 of 131072 cells, 32 / 4 heads,
    # head_dim 128) over an int8 cache, against the oracle
    inp = W.gather_inputs(1, 1, 32, 4, 128, 131072, 2048, 128, 1, device="cuda", int8=True)
    got = run_gpu(inp, torch.bfloat16, kernel=kernel)
    torch.cuda.synchronize()
    cpu = W.DecodeInputs(q=inp.q.cpu(), k=inp.k.cpu(), v=inp.v.cpu(),
                         kv_lengths=inp.kv_lengths.cpu(), n_q=1, causal=False, scale=inp.scale,
                         k_scale=inp.k_scale.cpu(), v_scale=inp.v_scale.cpu(),
                         idx=inp.idx.cpu())
    compare(got, run_oracle(cpu), torch.bfloat16, "int8 gather workload")


# -------------------------------------------------------------------- int8
@pytest.mark.parametrize("kernel", INT8_KERNELS)
@pytest.mark.parametrize("causal,n_q", [(False, 1), (True, 4)])
def test_int8_small(kernel, causal, n_q):
    inp = W.dense_inputs(3, n_q, 32, 8, 128, 640, [640, 200, 1], 24, causal, int8=True)
    check(inp, torch.bfloat16, kernel=kernel)
    check(inp, torch.float32, kernel=kernel)


@pytest.mark.parametrize("kernel", INT8_KERNELS)
@pytest.mark.parametrize("d", [128, 256])
def test_int8_poisoned_tail_scales(kernel, d):
    inp = W.dense_inputs(2, 1, 16, 4, d, 300, [150, 299], 25, False, int8=True, tail="nan")
    check(inp, torch.float32, kernel=kernel)


@pytest.mark.parametrize("ctas", [1, 3, 19, 300])
def test_int8_tensor_core_splits_and_32_rows(ctas):
    # 32 packed rows (8 heads per group x 4 causal rows), ragged lengths, the
    # segments cut into many split pieces
    inp = W.dense_inputs(3, 4, 32, 4, 128, 1500, [1500, 611, 129], 26, True, int8=True)
    check(inp, torch.float32, kernel=fd.FD_KERNEL_TC, num_ctas=ctas)
    check(inp, torch.bfloat16, kernel=fd.FD_KERNEL_TC, num_ctas=ctas)


@pytest.mark.parametrize("ctas", [1, 5, 64, 0])
@pytest.mark.parametrize("rows", [(8, 1, False), (4, 4, True), (8, 4, True)])
def test_int8_tensor_core_head_dim_256(ctas, rows):
    # head_dim 256 int8 caches on the tensor cores: 8 / 16 / 32 packed rows
    # (group x window), ragged lengths with a partial last tile, split pieces
    g, n_q, causal = rows
    inp = W.dense_inputs(3, n_q, 4 * g, 4, 256, 1100, [1100, 389, 77], 31, causal, int8=True)
    check(inp, torch.float32, kernel=fd.FD_KERNEL_TC, num_ctas=ctas)
    check(inp, torch.bfloat16, kernel=fd.FD_KERNEL_TC, num_ctas=ctas)


@pytest.mark.parametrize("d", [128, 256])
def test_int8_tensor_core_large_value_scales(d):
    # the tensor-core kernel multiplies in fp16: v scales up to 3000 (|v| up
    # to 3.8e5, inside the documented 4094 bound) and q entries near 6e4 stay
    # finite and match the oracle to fp16 / bf16 precision (relative check:
    # the outputs are of order 1e5)
    inp = W.dense_inputs(2, 1, 16, 4, d, 700, [700, 333], 33, False, int8=True)
    inp.v_scale = inp.v_scale * 1.0e5           # dequantised |v| ~ 3e5 at 3 sigma
    inp.q = inp.q.clone()
    inp.q[0, 0, 0, 0] = 60000.0                 # one large q entry (its bf16 value, 59904, is exact in fp16)
    ref = run_oracle(inp)
    dev = to_dev(inp)
    for od, tol in ((torch.float32, 1e-4), (torch.bfloat16, 4e-3)):
        got = run_gpu(dev, od, 0, fd.FD_KERNEL_TC).double().cpu()
        torch.cuda.synchronize()
        assert torch.isfinite(got).all()
        err = (got - ref.double()).abs().max() / ref.double().abs().max()
        assert err < tol, (od, float(err))


@pytest.mark.parametrize("ctas", [1, 7, 0])
@pytest.mark.parametrize("d", [128, 256])
@pytest.mark.parametrize("shape", [(2, 32, 1), (4, 64, 4), (6, 32, 4), (5, 48, 4), (3, 21, 1), (6, 18, 2)])
def test_int8_tensor_core_rows_in_parts(ctas, d, shape):
    # more than 32 packed rows (n_q x g = 64, 64, 48, 60, 63, 54): the
    # tensor-core kernel serves each kv head's query heads in 2 or 3 parts of
    # at most 32 rows; causal windows, ragged lengths down to one position
    n_q, Hq, Hkv = shape
    inp = W.dense_inputs(3, n_q, Hq, Hkv, d, 700, [700, 257, 1], 34, True, int8=True)
    check(inp, torch.float32, kernel=fd.FD_KERNEL_TC, num_ctas=ctas)
    check(inp, torch.bfloat16, kernel=fd.FD_KERNEL_TC, num_ctas=ctas)


def test_int8_rows_in_parts_need_workspace_segments():
    # 64 rows in 2 parts need 2 segments per (sequence, kv head): a workspace
    # with room for one per pair refuses the tensor-core kernel and sends
    # FD_KERNEL_AUTO to the CUDA-core kernel, which serves the rows in one pass
    inp = W.dense_inputs(2, 2, 32, 1, 128, 300, [300, 41], 35, True, int8=True)
    dev = to_dev(inp)
    ws = fd.Workspace(2, 64, 128, 1024)
    with pytest.raises(fd.FdError):
        run_gpu(dev, torch.float32, kernel=fd.FD_KERNEL_TC, workspace=ws)
    torch.cuda.synchronize()
    ws.reset()
    got = run_gpu(dev, torch.float32, workspace=ws)
    compare(got, run_oracle(inp), torch.float32, "int8 rows 64 auto, small workspace")
    ws.close()


def test_int8_tensor_core_rejects_unserved_shapes():
    # gather over an int8 cache with more than 32 rows (48 query heads on one
    # kv head): the tensor-core kernel declines and FD_KERNEL_AUTO takes the
    # CUDA-core one
    cpu = W.gather_inputs(1, 1, 48, 1, 128, 600, 200, 16, 27, int8=True)
    inp = to_dev(cpu)
    with pytest.raises(fd.FdError):
        run_gpu(inp, torch.float32, kernel=fd.FD_KERNEL_TC)
    compare(run_gpu(inp, torch.float32), run_oracle(cpu), torch.float32, "int8 gather rows 48 auto")


# ------------------------------------------------------------- CUDA graphs
@pytest.mark.parametrize("kernel", DENSE_KERNELS)
def test_graph_capture_and_replay_with_new_lengths(kernel):
    inp = W.dense_inputs(2, 4, 16, 4, 256, 1000, [1000, 1000], 26, True)
    dev = to_dev(inp)
    ws = fd.Workspace(16, 64, 256, 1024)
    out = torch.empty(dev.q.shape, dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fd.decode(dev.q, dev.k, dev.v, dev.kv_lengths, n_q=4, causal=True, scale=inp.scale,
                  out=out, kernel=kernel, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        fd.decode(dev.q, dev.k, dev.v, dev.kv_lengths, n_q=4, causal=True, scale=inp.scale,
                  out=out, kernel=kernel, workspace=ws)
    for lens in ([1000, 1000], [17, 999], [513, 4], [0, 640]):
        dev.kv_lengths.copy_(torch.tensor(lens, dtype=torch.int32))
        graph.replay()
        torch.cuda.synchronize()
        inp.kv_lengths = torch.tensor(lens, dtype=torch.int32)
        compare(out, run_oracle(inp), torch.float32, "graph replay %s" % lens)


# ------------------------------------------------------- full-size workloads
@pytest.mark.parametrize("kernel", DENSE_KERNELS)
@pytest.mark.parametrize("name", ["dense_1k", "mtp_verify", "gather", "ragged"])
def test_named_workload_full_size(kernel, name):
    inp = W.workload(name, seed=1)
    check(inp, torch.bfloat16, kernel=kernel)
    if name == "dense_1k":
        check(inp, torch.float32, kernel=kernel)
        poisoned = W.workload(name, seed=1, tail="nan")
        check(poisoned, torch.bfloat16, kernel=kernel)


@pytest.mark.parametrize("kernel", DENSE_KERNELS)
def test_mtp_verify_capacity_independent_output(kernel):
    # the MTP-verify shape at capacities 3000, 24007 and 131072 with the same
    # 3000 filled positions gives the same result
    base = W.workload("mtp_verify", seed=2)
    ref = run_oracle(base)
    outs = []
    for cap in (3000, 24007, 131072):
        inp = W.dense_inputs(1, 4, 16, 4, 256, cap, [3000], 2, True)
        inp.q.copy_(base.q)
        inp.k[:, :, :3000] = base.k[:, :, :3000]
        inp.v[:, :, :3000] = base.v[:, :, :3000]
        (_, _, _), got = check(inp, torch.float32, kernel=kernel, ref=ref)
        outs.append(got.cpu())
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])


@pytest.mark.parametrize("kernel", INT8_KERNELS)
def test_int8_workload_full_size_sampled(kernel):
    # full int8 workload (4 x 131072 tokens, 32/8 heads): generated on the GPU,
    # every output row checked against the oracle on the same bits
    inp = W.workload("int8", seed=1, device="cuda")
    got = run_gpu(inp, torch.bfloat16, kernel=kernel)
    torch.cuda.synchronize()
    cpu = W.DecodeInputs(q=inp.q.cpu(), k=inp.k.cpu(), v=inp.v.cpu(),
                         kv_lengths=inp.kv_lengths.cpu(), n_q=1, causal=False,
                         scale=inp.scale, k_scale=inp.k_scale.cpu(),
                         v_scale=inp.v_scale.cpu())
    compare(got, run_oracle(cpu), torch.bfloat16, "int8 full")


@pytest.mark.parametrize("kernel", INT8_KERNELS)
def test_int8_head_dim_256_full_size(kernel):
    # the int8 workload's shape at head_dim 256 (4 x 131072 tokens, 32 / 8
    # heads, 2.1 GB of codes): every output row against the oracle
    inp = W.dense_inputs(4, 1, 32, 8, 256, 131072, [131072] * 4, 2, False, device="cuda",
                         int8=True)
    got = run_gpu(inp, torch.bfloat16, kernel=kernel)
    torch.cuda.synchronize()
    cpu = W.DecodeInputs(q=inp.q.cpu(), k=inp.k.cpu(), v=inp.v.cpu(),
                         kv_lengths=inp.kv_lengths.cpu(), n_q=1, causal=False,
                         scale=inp.scale, k_scale=inp.k_scale.cpu(),
                         v_scale=inp.v_scale.cpu())
    compare(got, run_oracle(cpu), torch.bfloat16, "int8 d256 full")


# -------------------------------------------------- kernel choice by layout
def test_tensor_core_kernel_declines_unaligned_q():
    # q whose base is 2 bytes off a 16-byte boundary cannot be read through a
    # TMA map: the tensor-core kernel declines, AUTO takes the CUDA-core one
    inp = W.dense_inputs(2, 1, 8, 2, 128, 300, [300, 41], 29, False)
    dev = to_dev(inp)
    buf = torch.empty(dev.q.numel() + 1, dtype=torch.bfloat16, device="cuda")
    q = buf[1:].view(dev.q.shape)
    q.copy_(dev.q)
    assert q.data_ptr() % 16 != 0
    with pytest.raises(fd.FdError):
        fd.decode(q, dev.k, dev.v, dev.kv_lengths, n_q=1, scale=inp.scale,
                  out_dtype=torch.float32, kernel=fd.FD_KERNEL_TC)
    got = fd.decode(q, dev.k, dev.v, dev.kv_lengths, n_q=1, scale=inp.scale,
                    out_dtype=torch.float32)
    compare(got, run_oracle(inp), torch.float32, "unaligned q, auto")


def test_inputs_changed_in_place_between_calls():
    # the same tensors (so the same cached tensor maps) with new contents
    inp = W.dense_inputs(2, 4, 16, 4, 256, 900, [900, 333], 30, True)
    dev = to_dev(inp)
    ws = fd.Workspace(8, 16, 256, 1024)
    out = torch.empty(dev.q.shape, dtype=torch.float32, device="cuda")
    for step in range(3):
        fd.decode(dev.q, dev.k, dev.v, dev.kv_lengths, n_q=4, causal=True, scale=inp.scale,
                  out=out, workspace=ws, kernel=fd.FD_KERNEL_TC)
        torch.cuda.synchronize()
        compare(out, run_oracle(inp), torch.float32, "step %d" % step)
        g = torch.Generator().manual_seed(100 + step)
        inp.q = torch.randn(inp.q.shape, generator=g).to(torch.bfloat16)
        inp.k = torch.randn(inp.k.shape, generator=g).to(torch.bfloat16)
        dev.q.copy_(inp.q)
        dev.k.copy_(inp.k)
