"""Seeded synthetic inputs for triangular attention.

This module holds no arithmetic of the method: it only draws random tensors.
The same generator feeds the CUDA path and the FP64 oracle, so both see the
same BF16 values.

The pages measure on captured OpenFold3 activations that are not available,
so seeded synthetic tensors with the shapes and value distributions of the
pages' crop configurations stand in for them ("TurboPairFormer", Table 8 and
Figure 4 give the crop sizes 384/640/768 and head dimensions 16/32 with
B=1, N_o=N, H=4).

Draw order (one ``torch.Generator`` on the CPU, seeded): q, k, v, dO, bias,
then the mask.  Every normal draw is made in FP32 and rounded once to BF16.
The mask is additive BF16, 0 for a kept key and -inf for a masked key, with
shape [B, N_o, N].
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    N: int
    H: int
    D: int
    bias_std: float = 1.0
    mask: str = "none"          # "none" | "tail" | "random"
    mask_frac: float = 0.0
    peaky_p: float = 0.0        # probability that a bias entry is replaced by peaky_value
    peaky_value: float = 8.0

    @property
    def No(self) -> int:
        return self.N           # the method has N_o = N

    def describe(self) -> str:
        return (f"{self.name}: B={self.B} N=N_o={self.N} H={self.H} D={self.D} "
                f"bias~N(0,{self.bias_std:g}^2) mask={self.mask}:{self.mask_frac:g}"
                + (f" peaky p={self.peaky_p:g}->{self.peaky_value:g}" if self.peaky_p else ""))


# The five workload families (seven shapes) of the pages' crop sizes.
WORKLOADS = {
    "tiny48": Workload("tiny48", B=1, N=48, H=2, D=16),
    "crop384": Workload("crop384", B=1, N=384, H=4, D=32, bias_std=2.0, mask="tail", mask_frac=0.10),
    "crop640_d16": Workload("crop640_d16", B=1, N=640, H=4, D=16, mask="random", mask_frac=0.05),
    "crop640_h8d32": Workload("crop640_h8d32", B=1, N=640, H=8, D=32, mask="random", mask_frac=0.05),
    "crop768": Workload("crop768", B=1, N=768, H=4, D=32, mask="tail", mask_frac=0.08),
    "crop768_d16": Workload("crop768_d16", B=1, N=768, H=4, D=16, mask="tail", mask_frac=0.08),
    "long1024": Workload("long1024", B=2, N=1024, H=4, D=32, bias_std=4.0, mask="tail", mask_frac=0.10,
                         peaky_p=0.01, peaky_value=8.0),
}


def custom(B: int, N: int, H: int, D: int, name: str = "custom", No: Optional[int] = None, **kw) -> Workload:
    if No is not None and No != N:
        raise ValueError("the method has N_o = N")
    return Workload(name, B=B, N=N, H=H, D=D, **kw)


def make_inputs(w: Workload, seed: int = 0) -> dict:
    """Draw q, k, v, dO [B,N_o,H,N,D], bias [B,H,N,N] and mask [B,N_o,N]
    (or None) as CPU BF16 tensors."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    shp = (w.B, w.No, w.H, w.N, w.D)

    def normal(shape, std=1.0):
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        return x.to(torch.bfloat16)

    q = normal(shp)
    k = normal(shp)
    v = normal(shp)
    do = normal(shp)
    bias = torch.randn((w.B, w.H, w.N, w.N), generator=g, dtype=torch.float32)
    if w.bias_std != 1.0:
        bias.mul_(w.bias_std)
    if w.peaky_p > 0:
        hit = torch.rand(bias.shape, generator=g) < w.peaky_p
        bias[hit] = w.peaky_value
    bias = bias.to(torch.bfloat16)
    mask = None
    if w.mask == "tail":
        nm = int(w.mask_frac * w.N)
        mask = torch.zeros((w.B, w.No, w.N), dtype=torch.float32)
        if nm > 0:
            mask[:, :, w.N - nm:] = float("-inf")
        mask = mask.to(torch.bfloat16)
    elif w.mask == "random":
        drop = torch.rand((w.B, w.No, w.N), generator=g) < w.mask_frac
        full = drop.all(dim=-1)
        if bool(full.any()):
            # keep at least one key per row: re-open one random key
            idx = torch.randint(0, w.N, (int(full.sum()),), generator=g)
            rows = full.nonzero()
            for r, kk in zip(rows.tolist(), idx.tolist()):
                drop[r[0], r[1], kk] = False
        mask = torch.zeros((w.B, w.No, w.N), dtype=torch.float32)
        mask[drop] = float("-inf")
        mask = mask.to(torch.bfloat16)
    elif w.mask != "none":
        raise ValueError(w.mask)
    return {"q": q, "k": k, "v": v, "do": do, "bias": bias, "mask": mask}


def make_module_inputs(B: int, N: int, C: int, H: int, D: int, seed: int = 0, mask_frac: float = 0.0) -> dict:
    """Seeded inputs of the module around the core (CPU tensors): z and the
    incoming gradient d_out [B, N, N, C] BF16 (standard normal), LayerNorm
    scale 1 + 0.1 n and shift 0.1 n (FP32), W_in [C, 3HD + H] with entries
    n / sqrt(C) and W_o [HD, C] with entries n / sqrt(HD) (BF16), so that q,
    k, v and the bias channels have about unit variance, as the core's own
    synthetic inputs do.  Draw order: z, d_out, ln_w, ln_b, W_in, W_o.  With
    ``mask_frac`` > 0 the last ``int(mask_frac * N)`` keys of every slice are
    masked ([B, N, N] additive BF16, -inf), else the mask is None."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))

    def normal(shape, scale=1.0):
        return torch.randn(shape, generator=g, dtype=torch.float32) * scale

    F = 3 * H * D + H
    z = normal((B, N, N, C)).to(torch.bfloat16)
    d_out = normal((B, N, N, C)).to(torch.bfloat16)
    ln_w = 1.0 + normal((C,), 0.1)
    ln_b = normal((C,), 0.1)
    w_in = normal((C, F), C ** -0.5).to(torch.bfloat16)
    w_o = normal((H * D, C), (H * D) ** -0.5).to(torch.bfloat16)
    mask = None
    nm = int(mask_frac * N)
    if nm > 0:
        mask = torch.zeros((B, N, N), dtype=torch.float32)
        mask[:, :, N - nm:] = float("-inf")
        mask = mask.to(torch.bfloat16)
    return {"z": z, "d_out": d_out, "ln_w": ln_w, "ln_b": ln_b, "w_in": w_in, "w_o": w_o, "mask": mask,
            "H": H, "D": D}


def make_trimul_inputs(B: int, N: int, Cz: int, Ch: int, seed: int = 0, pad_frac: float = 0.0) -> dict:
    """Seeded inputs of the triangle multiplicative update (CPU tensors): z
    and d_out [B, N, N, C_z] BF16 (standard normal); LayerNorm scales
    1 + 0.1 n and shifts 0.1 n (FP32) for the input (C_z) and output (C_h)
    normalizations; W_p [C_z, 4 C_h + C_z] with entries n / sqrt(C_z) and W_o
    [C_h, C_z] with entries n / sqrt(C_h) (BF16).  Draw order: z, d_out,
    ln_in_w, ln_in_b, W_p, ln_out_w, ln_out_b, W_o.  With ``pad_frac`` > 0 the
    last ``int(pad_frac * N)`` tokens are padding: the multiplicative pair
    mask [B, N, N] (BF16) is 0 for every pair that touches one, else 1;
    otherwise the mask is None."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))

    def normal(shape, scale=1.0):
        return torch.randn(shape, generator=g, dtype=torch.float32) * scale

    z = normal((B, N, N, Cz)).to(torch.bfloat16)
    d_out = normal((B, N, N, Cz)).to(torch.bfloat16)
    ln_in_w = 1.0 + normal((Cz,), 0.1)
    ln_in_b = normal((Cz,), 0.1)
    w_p = normal((Cz, 4 * Ch + Cz), Cz ** -0.5).to(torch.bfloat16)
    ln_out_w = 1.0 + normal((Ch,), 0.1)
    ln_out_b = normal((Ch,), 0.1)
    w_o = normal((Ch, Cz), Ch ** -0.5).to(torch.bfloat16)
    mask = None
    npad = int(pad_frac * N)
    if npad > 0:
        keep = torch.ones(N)
        keep[N - npad:] = 0.0
        mask = (keep[:, None] * keep[None, :]).expand(B, N, N).contiguous().to(torch.bfloat16)
    return {"z": z, "d_out": d_out, "ln_in_w": ln_in_w, "ln_in_b": ln_in_b, "w_p": w_p, "ln_out_w": ln_out_w,
            "ln_out_b": ln_out_b, "w_o": w_o, "mask": mask}
