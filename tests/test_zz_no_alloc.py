"""fd_decode_noalloc: the decode entry point for callers that cannot allocate
device memory (their own allocator owns the GPU, or they run under a hard
memory cap).  It keeps its scratch in a fixed array inside libfd.so instead
of a workspace made with cudaMalloc.  This file runs last so that a failure
here never hides the other tests' results; it also passes on its own in a
fresh process."""
import ctypes

import pytest
import torch

from decode_attention_preallocated_gb300 import build as fdbuild
from decode_attention_preallocated_gb300 import fd
from decode_attention_preallocated_gb300 import workloads as W
from parity_util import compare, to_dev

pytestmark = pytest.mark.gpu


def call_noalloc(dev, out, num_ctas=0):
    tq, tk, tv, to = map(fd.as_fd_tensor, (dev.q, dev.k, dev.v, out))
    stream = torch.cuda.current_stream().cuda_stream
    return fd.lib().fd_decode_noalloc(ctypes.byref(tq), ctypes.byref(tk), ctypes.byref(tv),
                                      dev.kv_lengths.data_ptr(), dev.n_q, int(dev.causal),
                                      float(dev.scale), ctypes.byref(to), stream, num_ctas)


def test_noalloc_matches_fd_decode_on_two_calls_in_a_row():
    fdbuild.build()
    torch.cuda.set_device(0)
    inp = W.dense_inputs(2, 4, 16, 4, 256, 900, [900, 333], 31, True, tail="nan")
    dev = to_dev(inp)
    # the tail past each sequence's first length is NaN, so later lengths stay inside it
    for lens in ([900, 333], [5, 321]):
        dev.kv_lengths.copy_(torch.tensor(lens, dtype=torch.int32))
        ref = fd.decode(dev.q, dev.k, dev.v, dev.kv_lengths, n_q=4, causal=True,
                        scale=dev.scale, out_dtype=torch.float32)
        out = torch.full(dev.q.shape, float("nan"), dtype=torch.float32, device="cuda")
        assert call_noalloc(dev, out) == fd.FD_OK
        torch.cuda.synchronize()
        compare(out, ref, torch.float32, "noalloc vs fd_decode, lengths %s" % lens)


def test_noalloc_rejects_problems_beyond_its_scratch():
    fdbuild.build()
    # 64 query rows x d=256 per slot: 5000 (sequence, kv head) pairs exceed
    # the 4096-pair limit; the check runs before any launch
    q = torch.zeros((1, 1, 1, 256), dtype=torch.bfloat16, device="cuda")
    inp = W.DecodeInputs(q=q, k=torch.zeros((1, 1, 8, 256), dtype=torch.bfloat16, device="cuda"),
                         v=torch.zeros((1, 1, 8, 256), dtype=torch.bfloat16, device="cuda"),
                         kv_lengths=torch.ones(1, dtype=torch.int32, device="cuda"),
                         n_q=1, causal=False, scale=1.0)
    big = W.DecodeInputs(q=torch.zeros((5000, 1, 1, 256), dtype=torch.bfloat16, device="cuda"),
                         k=torch.zeros((5000, 1, 8, 256), dtype=torch.bfloat16, device="cuda"),
                         v=torch.zeros((5000, 1, 8, 256), dtype=torch.bfloat16, device="cuda"),
                         kv_lengths=torch.ones(5000, dtype=torch.int32, device="cuda"),
                         n_q=1, causal=False, scale=1.0)
    out = torch.empty((5000, 1, 1, 256), dtype=torch.float32, device="cuda")
    assert call_noalloc(big, out) == fd.FD_ERR_SCRATCH
    out1 = torch.empty((1, 1, 1, 256), dtype=torch.float32, device="cuda")
    assert call_noalloc(inp, out1, num_ctas=1 << 20) == fd.FD_ERR_SCRATCH
    assert call_noalloc(inp, out1) == fd.FD_OK
    torch.cuda.synchronize()
