"""Shared helpers for the tests: moving seeded inputs to the oracle and comparing results."""
import math

import numpy as np
import torch

import oracle

# tolerances of the operator's contract: bf16 I/O with fp32 accumulation, and fp32
TOL = {
    torch.bfloat16: {"o": 2e-2, "lse": 1e-2},
    torch.float32: {"o": 1e-5, "lse": 1e-5},
}


def cpu32(t):
    return None if t is None else t.detach().to("cpu").float().contiguous()


def oracle_full(a, rows=None):
    """Oracle (float64) on the whole problem of workload `a` (inputs taken from the tensors the
    kernel saw, copied to the CPU in [B, N, H, d] order)."""
    return oracle.attn_fwd(cpu32(a.q), cpu32(a.k), cpu32(a.v), bias=cpu32(a.bias),
                           kv_lens=None if a.kv_lens is None else a.kv_lens.cpu(),
                           causal=a.causal, scale=a.scale, rows=rows)


def empty_rows(a):
    """Boolean [B, H, Nq]: rows whose visible set is empty (ignoring bias -inf)."""
    lens = a.kv_len_list()
    e = np.zeros((a.B, a.H, a.Nq), bool)
    for b, n in enumerate(lens):
        for i in range(a.Nq):
            last = n - 1 if not a.causal else min(n - 1, i + n - a.Nq)
            e[b, :, i] = last < 0
    return e


def compare(o_gpu, lse_gpu, o_ref, lse_ref, dtype, empty=None, what=""):
    """Element-wise comparison within the contract's tolerance; empty rows bit-exact."""
    tol = TOL[dtype]
    o = o_gpu.detach().float().cpu().numpy().astype(np.float64)
    lse = lse_gpu.detach().float().cpu().numpy().astype(np.float64)
    assert o.shape == o_ref.shape and lse.shape == lse_ref.shape
    assert not np.any(np.isnan(o)), f"{what}: NaN in o"
    assert not np.any(np.isnan(lse)), f"{what}: NaN in lse"
    finite = np.isfinite(lse_ref)
    # rows whose reference lse is -inf are empty: exact +0.0 and -inf
    assert np.all(lse[~finite] == -np.inf), f"{what}: empty rows must have lse = -inf"
    o_empty = np.transpose(o, (0, 2, 1, 3))[~finite]  # [n_empty, dv]
    raw = o_gpu.detach().cpu()
    if raw.dtype == torch.bfloat16:
        bits = raw.view(torch.int16).numpy()
    else:
        bits = raw.view(torch.int32).numpy()
    bits_empty = np.transpose(bits, (0, 2, 1, 3))[~finite]
    assert np.all(bits_empty == 0), f"{what}: empty rows must be +0.0 exactly"
    if empty is not None:
        assert np.array_equal(~finite, empty), f"{what}: empty-row set differs"
    err_o = np.max(np.abs(o - o_ref)) if o.size else 0.0
    err_l = np.max(np.abs(lse[finite] - lse_ref[finite])) if finite.any() else 0.0
    assert err_o <= tol["o"], f"{what}: max |o - oracle| = {err_o:.3e} > {tol['o']}"
    assert err_l <= tol["lse"], f"{what}: max |lse - oracle| = {err_l:.3e} > {tol['lse']}"
    return err_o, err_l


def sample_rows(a, n_per_head=24, seed=0, heads=None):
    """Flat row indices (b*H + h)*Nq + i: the first and last rows of every tile edge plus a
    seeded random sample, for every (b, h) in `heads` (default all)."""
    rng = np.random.default_rng(seed)
    rows = []
    heads = heads if heads is not None else [(b, h) for b in range(a.B) for h in range(a.H)]
    for (b, h) in heads:
        base = (b * a.H + h) * a.Nq
        pick = {0, a.Nq - 1, min(127, a.Nq - 1), min(128, a.Nq - 1)}
        pick |= set(rng.integers(0, a.Nq, n_per_head).tolist())
        rows += [base + i for i in sorted(pick)]
    return np.asarray(rows, np.int64)


def gather_rows(o, lse, rows, H, Nq):
    """GPU outputs at flat rows -> (o [n, dv] float64, lse [n] float64)."""
    o = o.detach().float().cpu().numpy().astype(np.float64)
    lse = lse.detach().float().cpu().numpy().astype(np.float64)
    b = rows // (H * Nq)
    h = (rows // Nq) % H
    i = rows % Nq
    return o[b, i, h], lse[b, h, i]


def compare_rows(o_s, l_s, o_ref, l_ref, dtype, what=""):
    tol = TOL[dtype]
    finite = np.isfinite(l_ref)
    assert np.all(l_s[~finite] == -np.inf), what
    assert np.all(o_s[~finite] == 0.0), what
    err_o = np.max(np.abs(o_s - o_ref))
    err_l = np.max(np.abs(l_s[finite] - l_ref[finite])) if finite.any() else 0.0
    assert err_o <= tol["o"], f"{what}: max |o - oracle| = {err_o:.3e}"
    assert err_l <= tol["lse"], f"{what}: max |lse - oracle| = {err_l:.3e}"
    return err_o, err_l
