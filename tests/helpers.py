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


# Gradient bound of the bf16 backward.  The kernels round P and dS to bf16 before the products
# that form dV, dK and dQ (a relative error of at most 2^-9 per term), accumulate in fp32 and
# store the gradients in bf16 (2^-9 again).  An element of a gradient is a sum over rows or
# keys of such rounded terms whose errors have random signs, so its error is about 2^-9 times
# the root sum of squares of the terms, which is of the size of the gradient row it belongs
# to; the stored value adds 2^-9 of the element itself.  One more error does not cancel:
# c_i = dO_i . O_i is formed from the O the forward stored in bf16 (its rounding, 2^-9, plus
# the forward's own error of the same order), so |dc_i| <= 2^-8 sum_c |dO_ic O_ic|, and since
# the weights of a row sum to 1 that error reaches dQ_i as -scale dc_i sum_j p_ij k_j, at most
# scale |dc_i| max_j |k_jd| in dimension d.  It matters where dQ_i itself nearly cancels (a row
# that sees one or two keys).  A backward that rounds exactly where the kernels round
# (tests/test_grad_bound.py) stays under 0.031 x the row's RMS beyond 2^-6 |ref| and the c
# term, with a relative Frobenius error of 2.2e-3 to 2.8e-3 per tensor.  The bound keeps a
# margin of 2 to 4 over both:
#   |g - ref| <= GRAD_RTOL |ref| + GRAD_ATOL_ROW rms(ref row) + (dQ only) the c term
#   ||g - ref|| / ||ref|| <= GRAD_FRO
# where a "row" is the head-dimension vector of one query (dQ) or one key (dK, dV) of one
# (b, h).  A floor of GRAD_ATOL_TENSOR rms(ref) covers elements whose exact value vanishes by
# cancellation (a key that every row sees alone: p = 1 and dS = dP - c = 0), where the kernel
# keeps the fp32 residue of the cancelling sums, some 1e-5.
GRAD_RTOL = 2.0 ** -6
GRAD_ATOL_ROW = 2.0 ** -4
GRAD_ATOL_TENSOR = 2.0 ** -10
GRAD_FRO = 1e-2


def dq_c_term(dout, o, k, scale, kv_lens=None):
    """[B, Nq, H, dk] float64: the part of the dQ bound that the bf16 O's rounding in
    c_i = dO_i . O_i can reach (see above).  dout, o [B, Nq, H, dv]; k [B, Nk, H, dk]; keys
    past kv_lens (or non-finite) are left out of the maximum."""
    def arr(t):
        return t.detach().float().cpu().numpy().astype(np.float64) if torch.is_tensor(t) else np.asarray(t, np.float64)
    g, oo, kk = arr(dout), arr(o), arr(k)
    dc = 2.0 ** -8 * np.sum(np.abs(g * oo), axis=-1, keepdims=True)        # [B, Nq, H, 1]
    ak = np.where(np.isfinite(kk), np.abs(kk), 0.0)
    if kv_lens is not None:
        lens = [int(x) for x in (kv_lens.tolist() if torch.is_tensor(kv_lens) else kv_lens)]
        for b, n in enumerate(lens):
            ak[b, max(0, n):] = 0.0
    kmax = ak.max(axis=1, initial=0.0)[:, None]                          # [B, 1, H, dk]
    return scale * dc * kmax


def grad_bound_violations(got, ref, extra=None):
    """(number of elements over the per-element bound, relative Frobenius error) of a gradient
    `got` against the float64 `ref`, both [..., d] (got may be a bf16 tensor or an array);
    `extra` (broadcastable to ref) is added to the per-element limit (the dQ c term)."""
    g = got.detach().float().cpu().numpy().astype(np.float64) if torch.is_tensor(got) else np.asarray(got, np.float64)
    r = np.asarray(ref, np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    if r.size == 0:
        return 0, 0.0
    err = np.abs(g - r)
    rms_row = np.sqrt(np.mean(r * r, axis=-1, keepdims=True))
    lim = GRAD_RTOL * np.abs(r) + GRAD_ATOL_ROW * rms_row + GRAD_ATOL_TENSOR * float(np.sqrt(np.mean(r * r)))
    if extra is not None:
        lim = lim + extra
    nref = float(np.linalg.norm(r))
    fro = float(np.linalg.norm(g - r)) / nref if nref > 0 else float(np.linalg.norm(g))
    bad = int(np.count_nonzero(~(err <= lim)))
    return bad, fro


def check_grad(got, ref, what, zero=None, extra=None):
    """Gradient parity within the bound above; `zero` [B, N] marks rows (keys or query rows)
    that must be +0.0 bit for bit; `extra` is the dQ c term (dq_c_term) for dQ."""
    g = got.detach().float().cpu().numpy()
    assert np.all(np.isfinite(g)), f"{what}: non-finite"
    bad, fro = grad_bound_violations(got, ref, extra)
    assert bad == 0, f"{what}: {bad} elements over the per-element gradient bound (relative Frobenius {fro:.2e})"
    assert fro <= GRAD_FRO, f"{what}: relative Frobenius error {fro:.3e} > {GRAD_FRO}"
    if zero is not None:
        bits = got.detach().cpu().view(torch.int16).numpy()
        assert np.all(bits[zero] == 0), f"{what}: rows that must be +0.0 are not"
