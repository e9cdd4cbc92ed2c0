"""Failure detection on the GPU without a GPU fault.

Every internal wait of the tensor-core kernel is bounded; one that runs out
sets FD_DEV_INTERNAL in the workspace status word, records where it waited
(fd_get_device_diagnostics) and lets the launch end, so the context stays
usable.  Here the wait is made to run out on purpose: the workspace's
completion counters are preset to a negative value (what a launch aborted
part-way can leave behind), so the blocks that share the merge of a split
segment wait for a count that never comes.  The host reads the status, resets
the workspace (fd_workspace_reset) and the next call matches the fp64 oracle
again."""
import time

import pytest
import torch

from decode_attention_preallocated_gb300 import fd
from decode_attention_preallocated_gb300 import workloads as W
from parity_util import compare, run_oracle, to_dev

pytestmark = pytest.mark.gpu

# wait ids recorded by the tensor-core kernel for the shared merge: 14 = the
# barrier of the softmax warps, 15 = the wait for every piece's count
SHARED_MERGE_WAITS = (14, 15)


def mtp_inputs():
    # the MTP-verify shape: 4 causal rows, 16 / 4 heads, head_dim 256, 3000
    # filled positions; it runs the cooperative launch whose blocks share the
    # merges of the few split segments
    inp = W.dense_inputs(1, 4, 16, 4, 256, 4096, [3000], 41, True, tail="nan")
    return inp, to_dev(inp)


def call(dev, ws, wait_limit_us=0):
    return fd.decode(dev.q, dev.k, dev.v, dev.kv_lengths, n_q=dev.n_q, causal=True,
                     scale=dev.scale, out_dtype=torch.float32, kernel=fd.FD_KERNEL_TC,
                     workspace=ws, wait_limit_us=wait_limit_us)


def test_a_short_wait_limit_leaves_normal_calls_alone():
    torch.cuda.set_device(0)
    inp, dev = mtp_inputs()
    ws = fd.Workspace(4, 16, 256, 2048)
    out = call(dev, ws, wait_limit_us=20000)
    torch.cuda.synchronize()
    assert ws.device_status() == 0
    compare(out, run_oracle(inp), torch.float32, "20 ms wait limit")
    ws.close()


def test_stale_counters_make_a_bounded_wait_give_up_and_reset_recovers():
    torch.cuda.set_device(0)
    inp, dev = mtp_inputs()
    ref = run_oracle(inp)
    ws = fd.Workspace(4, 16, 256, 2048)
    ws.fill_counters(-1000)
    t0 = time.perf_counter()
    call(dev, ws, wait_limit_us=20000)
    torch.cuda.synchronize()            # the launch ends: no wait is unbounded
    elapsed = time.perf_counter() - t0
    st = ws.diagnostics()
    assert st[0] & fd.FD_DEV_INTERNAL, "status %r" % (st,)
    assert st[1] in SHARED_MERGE_WAITS, "first wait that gave up: %d" % st[1]
    assert st[4 + 3 * 2] in SHARED_MERGE_WAITS, "softmax role's wait: %d" % st[4 + 3 * 2]
    assert elapsed < 10.0, "the launch took %.1f s to give up" % elapsed
    # the status word is sticky until the workspace is reset
    assert ws.device_status() & fd.FD_DEV_INTERNAL
    ws.reset()
    assert ws.device_status() == 0
    for _ in range(2):   # twice: the counters are back to self-resetting
        out = call(dev, ws)
        torch.cuda.synchronize()
        assert ws.device_status() == 0
        compare(out, ref, torch.float32, "after fd_workspace_reset")
    ws.close()
