"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
the fp64 oracle on the same seeded inputs, and compare with the tolerances
the decode-attention contract states (bf16 output: max |err| <= 1e-2 and
mean |err| <= 1e-3; fp32 output: max |err| <= 2e-3)."""
from __future__ import annotations

import torch

import oracle
from decode_attention_preallocated_gb300 import fd

TOL = {torch.bfloat16: (1e-2, 1e-3), torch.float32: (2e-3, 2e-3)}


def to_dev(inp, device="cuda"):
    """Copy a DecodeInputs to the GPU (keeping strided cache layouts)."""
    import copy
    out = copy.copy(inp)
    for name in ("q", "kv_lengths", "k_scale", "v_scale", "idx", "block_table"):
        t = getattr(inp, name)
        if t is not None:
            setattr(out, name, t.to(device))
    for name in ("k", "v"):
        t = getattr(inp, name)
        if t.is_contiguous():
            setattr(out, name, t.to(device))
        else:
            # token-major view [B, cap, Hkv, d] seen as [B, Hkv, cap, d]
            base = t.transpose(1, 2).contiguous().to(device)
            setattr(out, name, base.transpose(1, 2))
    return out


def run_gpu(inp, out_dtype=torch.bfloat16, num_ctas=0, kernel=fd.FD_KERNEL_AUTO,
            workspace=None):
    """One call through the C ABI.  Without an explicit workspace the call gets
    a fresh one, and afterwards its status word must not report an internal
    error (a bounded wait that gave up)."""
    own = workspace is None
    if own:
        B, n_q, Hq, d = inp.q.shape
        Hkv = inp.k.shape[1]
        workspace = fd.Workspace(B * n_q * Hkv, min(64, (Hq // Hkv) * n_q), 256,
                                 max(2048, num_ctas))
    if inp.block_table is not None:
        out = fd.decode_paged(inp.q, inp.k, inp.v, inp.block_table, inp.kv_lengths,
                              n_q=inp.n_q, causal=inp.causal, scale=inp.scale,
                              k_scale=inp.k_scale, v_scale=inp.v_scale, out_dtype=out_dtype,
                              num_ctas=num_ctas, kernel=kernel, workspace=workspace)
    elif inp.idx is not None:
        out = fd.decode_gather(inp.q, inp.k, inp.v, inp.idx, scale=inp.scale,
                               out_dtype=out_dtype, num_ctas=num_ctas, kernel=kernel,
                               workspace=workspace, k_scale=inp.k_scale, v_scale=inp.v_scale)
    elif inp.k.dtype == torch.int8:
        out = fd.decode_int8(inp.q, inp.k, inp.v, inp.k_scale, inp.v_scale,
                             inp.kv_lengths, n_q=inp.n_q, causal=inp.causal,
                             scale=inp.scale, out_dtype=out_dtype, num_ctas=num_ctas,
                             kernel=kernel, workspace=workspace)
    else:
        out = fd.decode(inp.q, inp.k, inp.v, inp.kv_lengths, n_q=inp.n_q,
                        causal=inp.causal, scale=inp.scale, out_dtype=out_dtype,
                        num_ctas=num_ctas, kernel=kernel, workspace=workspace)
    if own:
        torch.cuda.synchronize()
        st = workspace.diagnostics()
        assert not st[0] & fd.FD_DEV_INTERNAL, (
            "kernel %d reported an internal error: wait site %d, tile %d, piece %d"
            % (kernel, st[1], st[2], st[3]))
        workspace.close()
    return out


def run_oracle(inp):
    if inp.block_table is not None:
        return torch.from_numpy(oracle.paged(inp.q, inp.k, inp.v, inp.block_table.cpu(),
                                             inp.kv_lengths.cpu(), inp.n_q, inp.causal,
                                             inp.scale, inp.k_scale, inp.v_scale))
    if inp.idx is not None:
        return torch.from_numpy(oracle.gather(inp.q, inp.k, inp.v, inp.idx, inp.scale,
                                              inp.k_scale, inp.v_scale))
    lens = inp.kv_lengths.cpu()
    return torch.from_numpy(oracle.dense(inp.q, inp.k, inp.v, lens, inp.n_q, inp.causal,
                                         inp.scale, inp.k_scale, inp.v_scale))


def bf16_half_ulp(x: torch.Tensor) -> torch.Tensor:
    """Half a bf16 ulp at |x| (the largest error of a correctly rounded store)."""
    _, e = torch.frexp(x.abs())
    half = torch.ldexp(torch.ones_like(x), (e - 9).to(torch.int32))
    return torch.where(x == 0, torch.zeros_like(x), half)


def compare(got, ref, out_dtype, what=""):
    """Element-by-element check; returns (max abs, mean abs, normalised).

    For bf16 outputs the bound applies on top of the output's own rounding:
    |got - ref| <= 1e-2 + half a bf16 ulp of ref (an exactly computed value
    rounded to bf16 is already 0.0156 away from the fp64 answer when
    |ref| >= 4)."""
    g = got.detach().double().cpu()
    r = ref.double().cpu()
    assert g.shape == r.shape, (g.shape, r.shape)
    assert torch.isfinite(g).all(), "%s: non-finite output" % what
    err = (g - r).abs()
    mx, mean = float(err.max()), float(err.mean())
    norm = mx / max(float(r.abs().max()), 1e-30)
    tmax, tmean = TOL[out_dtype]
    slack = bf16_half_ulp(r) if out_dtype == torch.bfloat16 else torch.zeros_like(r)
    excess = float((err - slack).max())
    assert excess <= tmax, "%s: max abs err %.3e (beyond output rounding %.3e) > %.1e (mean %.3e)" % (
        what, mx, excess, tmax, mean)
    assert mean <= tmean, "%s: mean abs err %.3e > %.1e" % (what, mean, tmean)
    return mx, mean, norm
