"""fd_decode_noalloc: the decode entry point for callers that cannot allocate
device memory (their own allocator owns the GPU, they run under a hard
memory cap, or they are a plugin that may not allocate after start-up).  It
keeps its scratch in a fixed array inside libfd.so instead of a workspace
made with cudaMalloc.  Its output is checked against the fp64 oracle.  This
file runs last so that a failure here never hides the other tests' results;
it also passes on its own in a fresh process."""
import ctypes

import pytest
import torch

from decode_attention_preallocated_gb300 import build as fdbuild
from decode_attention_preallocated_gb300 import fd
from decode_attention_preallocated_gb300 import workloads as W
from parity_util import compare, run_oracle, to_dev

pytestmark = pytest.mark.gpu


def call_noalloc(dev, out, num_ctas=0):
    tq, tk, tv, to = map(fd.as_fd_tensor, (dev.q, dev.k, dev.v, out))
    stream = torch.cuda.current_stream().cuda_stream
    return fd.lib().fd_decode_noalloc(ctypes.byref(tq), ctypes.byref(tk), ctypes.byref(tv),
                                      dev.kv_lengths.data_ptr(), dev.n_q, int(dev.causal),
                                      float(dev.scale), ctypes.byref(to), stream, num_ctas)


def zeros_problem(B, Hq, Hkv, n_q, d=256, cap=8):
    z = lambda *s: torch.zeros(s, dtype=torch.bfloat16, device="cuda")  # noqa: E731
    return W.DecodeInputs(q=z(B, n_q, Hq, d), k=z(B, Hkv, cap, d), v=z(B, Hkv, cap, d),
                          kv_lengths=torch.ones(B, dtype=torch.int32, device="cuda"),
                          n_q=n_q, causal=False, scale=1.0)


def test_noalloc_matches_the_oracle_on_two_calls_in_a_row():
    fdbuild.build()
    torch.cuda.set_device(0)
    inp = W.dense_inputs(2, 4, 16, 4, 256, 900, [900, 333], 31, True, tail="nan")
    dev = to_dev(inp)
    # the tail past each sequence's first length is NaN, so later lengths stay inside it
    for lens in ([900, 333], [5, 321]):
        inp.kv_lengths = torch.tensor(lens, dtype=torch.int32)
        dev.kv_lengths.copy_(inp.kv_lengths)
        ref = run_oracle(inp)
        for out_dtype in (torch.float32, torch.bfloat16):
            out = torch.full(dev.q.shape, float("nan"), dtype=out_dtype, device="cuda")
            assert call_noalloc(dev, out) == fd.FD_OK
            torch.cuda.synchronize()
            compare(out, ref, out_dtype, "noalloc vs oracle, lengths %s, %s" % (lens, out_dtype))


def test_noalloc_takes_no_device_memory():
    fdbuild.build()
    torch.cuda.set_device(0)
    dev = to_dev(W.workload("dense_1k", seed=2))
    out = torch.empty(dev.q.shape, dtype=torch.bfloat16, device="cuda")
    assert call_noalloc(dev, out) == fd.FD_OK        # the first call loads the module
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        assert call_noalloc(dev, out) == fd.FD_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, "free device memory changed by %d bytes" % (free0 - free1)


def test_noalloc_rejects_problems_beyond_its_scratch():
    fdbuild.build()
    # 5000 (sequence, kv head) pairs of one query row: past the limit of 4096
    # pairs; the check runs before any launch
    big = zeros_problem(5000, 1, 1, 1)
    out = torch.empty(big.q.shape, dtype=torch.float32, device="cuda")
    assert call_noalloc(big, out) == fd.FD_ERR_SCRATCH
    # 200 pairs of 64 query rows x head_dim 256: within the pair limit, but
    # their split partials (201 slots of 64 x 256 floats) exceed the 8 MiB
    wide = zeros_problem(200, 64, 1, 1)
    out = torch.empty(wide.q.shape, dtype=torch.float32, device="cuda")
    assert call_noalloc(wide, out) == fd.FD_ERR_SCRATCH
    # one pair fits, but not an explicit block count of 2^20
    one = zeros_problem(1, 1, 1, 1)
    out1 = torch.empty(one.q.shape, dtype=torch.float32, device="cuda")
    assert call_noalloc(one, out1, num_ctas=1 << 20) == fd.FD_ERR_SCRATCH
    assert call_noalloc(one, out1) == fd.FD_OK
    torch.cuda.synchronize()
