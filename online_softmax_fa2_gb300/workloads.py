"""Seeded synthetic inputs for attention forward and split-KV decode.

This module holds no attention arithmetic: it only draws tensors.  The GPU tests, the
benchmark and the oracle checks all take their inputs from here, so the kernel and the
oracle always see the same (already rounded) values.

Five standard workloads (names are what they are, with their sizes):

  fp32_b1_h1_n128_d64          fp32, B=1, H=1, Nq=Nk=128, d=64, no mask, seed 0
  bf16_causal_b4_h16_n2048_d128  bf16, B=4, H=16, N=2048, d=128, causal
  bf16_padbias_b8_h8_n1024_dk192_dv128  bf16, B=8, H=8, N=1024, dk=192, dv=128,
                               kv_len ~ U{0..1024} (kv_len[0]=0, kv_len[7]=1024 forced),
                               fp32 bias ~ N(0,1) at visible positions
  bf16_causal_b1_h32_n16384_d128  bf16, B=1, H=32, N=16384, d=128, causal, one key per row
                               whose logit is raised by +8 (through q, see below)
  bf16_decode_b64_h32_l8192_d128  bf16 decode, B=64, H=32, Nq=1, cache 8192,
                               kv_len ~ U{1..8192} (kv_len[0]=1, kv_len[63]=8192), 16 splits
                               (decode(..., nq=4, causal=True): four query rows per sequence,
                               aligned to its end)

Layouts: q, o [B, N, H, d] (b, n, h, d order); k, v [B, N, H, d] for prefill and a
[B, H, L, d] cache for decode (passed to the library as strided views); bias [B, H, Nq, Nk]
fp32; kv_lens int32 [B].

"poison" (default on) writes NaN into every key/value row past a sequence's kv_len and into
the bias at every masked position.  A correct kernel never lets a masked position reach the
result, so poisoning must not change a single bit of the output.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch


@dataclass
class Attn:
    name: str
    dtype: torch.dtype
    B: int
    H: int
    Nq: int
    Nk: int
    dk: int
    dv: int
    causal: bool
    scale: float
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    bias: Optional[torch.Tensor] = None
    kv_lens: Optional[torch.Tensor] = None
    num_splits: int = 0
    meta: dict = field(default_factory=dict)

    def kv_len_list(self):
        if self.kv_lens is None:
            return [self.Nk] * self.B
        return [int(x) for x in self.kv_lens.tolist()]

    def visible_pairs(self) -> int:
        """Number of (query, key) pairs the mask leaves visible (bias -inf not counted)."""
        tot = 0
        for n in self.kv_len_list():
            if self.causal:
                for i in range(self.Nq):
                    tot += max(0, min(n, i + n - self.Nq + 1))
            else:
                tot += self.Nq * n
        return tot * self.H

    def flops(self) -> int:
        """Algorithmic FLOPs: 2*dk (QK^T) + 2*dv (PV) per visible pair."""
        return self.visible_pairs() * 2 * (self.dk + self.dv)

    def kv_bytes(self) -> int:
        """Key and value bytes a decode must read: visible keys only."""
        es = torch.tensor([], dtype=self.dtype).element_size()
        return sum(self.kv_len_list()) * self.H * (self.dk + self.dv) * es

    def algo_bytes(self) -> int:
        """Bytes a forward must move at the least: q, the key and value rows of each sequence's
        key length, the bias at visible positions (fp32), o, and lse (fp32)."""
        es = torch.tensor([], dtype=self.dtype).element_size()
        q_o = self.B * self.Nq * self.H * (self.dk + self.dv) * es
        bias = 4 * self.visible_pairs() if self.bias is not None else 0
        return q_o + self.kv_bytes() + bias + 4 * self.B * self.H * self.Nq


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def randn(shape, gen, device, dtype):
    """N(0,1) draws in fp32, rounded once to dtype."""
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(dtype)


def make_prefill(B, H, Nq, Nk, dk, dv, dtype=torch.bfloat16, causal=False, bias=False,
                 kv_lens=None, scale=None, seed=0, device="cpu", poison=True, name=None,
                 bias_mask_p=0.0):
    """Generic prefill inputs.  kv_lens: None or a list of B ints.  bias_mask_p: fraction
    of visible positions whose bias is set to -inf (an explicit mask)."""
    g = _gen(device, seed)
    q = randn((B, Nq, H, dk), g, device, dtype)
    k = randn((B, Nk, H, dk), g, device, dtype)
    v = randn((B, Nk, H, dv), g, device, dtype)
    kvl = None
    if kv_lens is not None:
        kvl = torch.tensor(list(kv_lens), dtype=torch.int32, device=device)
    b = None
    if bias:
        b = torch.randn((B, H, Nq, Nk), generator=g, device=device, dtype=torch.float32)
        if bias_mask_p > 0:
            u = torch.rand((B, H, Nq, Nk), generator=g, device=device)
            b = torch.where(u < bias_mask_p, torch.full_like(b, -math.inf), b)
    if poison:
        _poison(q, k, v, b, kvl, causal, Nq, Nk, seq_dim=1)
    return Attn(name or f"prefill_b{B}_h{H}_nq{Nq}_nk{Nk}_dk{dk}_dv{dv}", dtype, B, H, Nq, Nk,
                dk, dv, causal, float(scale if scale is not None else 1.0 / math.sqrt(dk)),
                q, k, v, b, kvl)


def _poison(q, k, v, bias, kvl, causal, Nq, Nk, seq_dim):
    """NaN into key/value rows past kv_len and into the bias at masked positions."""
    if kvl is None and not causal:
        return
    dev = k.device
    lens = kvl.to(torch.int64) if kvl is not None else torch.full((k.shape[0],), Nk,
                                                                   dtype=torch.int64, device=dev)
    j = torch.arange(Nk, device=dev)
    pad = j[None, :] >= lens[:, None]                       # [B, Nk]
    if kvl is not None:
        m = pad.view(k.shape[0], Nk, 1, 1) if seq_dim == 1 else pad.view(k.shape[0], 1, Nk, 1)
        k.masked_fill_(m, float("nan"))
        v.masked_fill_(m, float("nan"))
    if bias is not None:
        i = torch.arange(Nq, device=dev)
        masked = pad[:, None, None, :].expand(bias.shape[0], 1, Nq, Nk)
        if causal:
            later = j[None, None, :] > (i[None, :, None] + lens[:, None, None] - Nq)  # [B,Nq,Nk]
            masked = masked | later[:, None, :, :]
        bias.masked_fill_(masked.expand_as(bias), float("nan"))


def fp32_small(device="cpu", seed=0):
    return make_prefill(1, 1, 128, 128, 64, 64, torch.float32, seed=seed, device=device,
                        name="fp32_b1_h1_n128_d64")


def causal_2k(device="cpu", seed=1, d=128, bias=False, B=4, H=16):
    """The 2k causal workload (B4 H16 d128); d, bias, B and H give its variants."""
    name = f"bf16_causal_b{B}_h{H}_n2048_d{d}" + ("_bias" if bias else "")
    return make_prefill(B, H, 2048, 2048, d, d, torch.bfloat16, causal=True, bias=bias, seed=seed,
                        device=device, name=name)


def padded_bias(device="cpu", seed=2, poison=True):
    g = _gen("cpu", seed + 1000)
    lens = torch.randint(0, 1025, (8,), generator=g).tolist()
    lens[0], lens[7] = 0, 1024  # one fully empty sequence and one full one, always
    a = make_prefill(8, 8, 1024, 1024, 192, 128, torch.bfloat16, bias=True, kv_lens=lens,
                     seed=seed, device=device, poison=poison,
                     name="bf16_padbias_b8_h8_n1024_dk192_dv128")
    return a


def long_causal(device="cpu", seed=4, B=1, H=32, N=16384, d=128):
    """Causal prefill with one key per row whose logit is raised by exactly +8 before
    rounding: for each (h, i) draw j* ~ U{0..i} and, in fp32 before the bf16 cast, add
    (8/scale) * k_j* / |k_j*|^2 to q_i (k_j* taken as the rounded key)."""
    g = _gen(device, seed)
    scale = 1.0 / math.sqrt(d)
    q32 = torch.randn((B, N, H, d), generator=g, device=device, dtype=torch.float32)
    k = randn((B, N, H, d), g, device, torch.bfloat16)
    v = randn((B, N, H, d), g, device, torch.bfloat16)
    u = torch.rand((B, N, H), generator=g, device=device, dtype=torch.float64)
    i = torch.arange(N, device=device, dtype=torch.float64)[None, :, None]
    jstar = torch.clamp((u * (i + 1)).floor().to(torch.int64), max=N - 1)   # U{0..i}
    kf = k.float()
    idx = jstar[..., None].expand(B, N, H, d)
    kj = torch.gather(kf, 1, idx)                                          # k_{j*(i)}
    q32 += (8.0 / scale) * kj / (kj * kj).sum(-1, keepdim=True)
    q = q32.to(torch.bfloat16)
    del q32, kj, kf, idx
    return Attn(f"bf16_causal_b{B}_h{H}_n{N}_d{d}", torch.bfloat16, B, H, N, N, d, d, True,
                scale, q, k, v, meta={"jstar": jstar})


def decode(device="cpu", seed=5, B=64, H=32, L=8192, d=128, num_splits=16, poison=True,
           lens=None, nq=1, causal=False):
    """Split-KV decode: nq query rows per (b, h) (1 for one decode step; a few for several
    tokens of a sequence at once, with causal=True aligning them to the end of the
    sequence) against a [B, H, L, d] cache."""
    if lens is None:
        gl = _gen("cpu", seed + 1000)
        lens = torch.randint(1, L + 1, (B,), generator=gl).tolist()
        if B >= 2:
            lens[0], lens[B - 1] = 1, L
    g = _gen(device, seed)
    q = randn((B, nq, H, d), g, device, torch.bfloat16)
    kc = randn((B, H, L, d), g, device, torch.bfloat16)
    vc = randn((B, H, L, d), g, device, torch.bfloat16)
    kvl = torch.tensor(lens, dtype=torch.int32, device=device)
    if poison:
        j = torch.arange(L, device=device)
        pad = (j[None, :] >= kvl.to(torch.int64)[:, None]).view(B, 1, L, 1)
        kc.masked_fill_(pad, float("nan"))
        vc.masked_fill_(pad, float("nan"))
    # the library takes [B, N, H, d]-ordered strided views; the cache is [B, H, L, d] in memory
    k = kc.permute(0, 2, 1, 3)
    v = vc.permute(0, 2, 1, 3)
    name = f"bf16_decode_b{B}_h{H}_l{L}_d{d}" + (f"_nq{nq}" if nq > 1 else "") + ("_causal" if causal else "")
    return Attn(name, torch.bfloat16, B, H, nq, L, d, d, causal, 1.0 / math.sqrt(d), q, k, v, None,
                kvl, num_splits)


STANDARD = {
    "fp32_b1_h1_n128_d64": fp32_small,
    "bf16_causal_b4_h16_n2048_d128": causal_2k,
    "bf16_padbias_b8_h8_n1024_dk192_dv128": padded_bias,
    "bf16_causal_b1_h32_n16384_d128": long_causal,
    "bf16_decode_b64_h32_l8192_d128": decode,
}


def dropout_keep(B, H, Nq, Nk, p_drop, seed=0, device="cpu"):
    """Seeded keep mask [B, H, Nq, Nk] (bool): each position kept with probability 1 - p_drop."""
    g = _gen("cpu", seed + 2000)
    keep = torch.rand((B, H, Nq, Nk), generator=g) >= p_drop
    return keep.to(device)


def pack_keep_mask(keep):
    """Bit-packed keep mask for attn_fwd: uint8 [B, H, Nq, 16 * ceil(Nk / 128)], bit (j % 8) of
    byte j // 8 of a row = key j kept (rows padded with zero bytes to whole 128-key tiles)."""
    B, H, Nq, Nk = keep.shape
    nb = 16 * ((Nk + 127) // 128)
    bits = torch.zeros((B, H, Nq, nb * 8), dtype=torch.uint8, device=keep.device)
    bits[..., :Nk] = keep.to(torch.uint8)
    weights = torch.tensor([1, 2, 4, 8, 16, 32, 64, 128], dtype=torch.uint8, device=keep.device)
    return (bits.view(B, H, Nq, nb, 8) * weights).sum(-1).to(torch.uint8)
