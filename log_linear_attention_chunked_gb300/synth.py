"""Seeded synthetic inputs for log-linear attention.

This module holds no arithmetic of the method: it only draws random tensors
with the shapes and distributions of the workloads below.  Both the GPU path
and the CPU oracle consume the tensors it returns (the oracle as a float64
copy of the values actually fed to the GPU, bf16-rounded where the GPU path
takes bf16), so it is the one piece of code the two sides share.

Every (tensor, batch row, head) slice has its own seed, a 64-bit mix of the
workload seed, the tensor name and (b, h), so any slice can be regenerated on
its own.  Draws happen in float32 on the requested device with a
``torch.Generator`` of that device; a CPU draw and a CUDA draw of the same
slice differ, so a test always feeds both sides from one draw.
"""

from __future__ import annotations

import math
import zlib

import torch

# Workloads.  Distributions: q, k ~ N(0,1)/sqrt(dk); v ~ N(0,1);
# log_alpha = -softplus(N(0,1) + shift); lam = softplus(N(0,1));
# Gated DeltaNet: k ~ N(0,1) then L2-normalised per token and head,
# beta = sigmoid(N(0,1)).  Backward: the upstream gradient dout ~ N(0,1).
WORKLOADS = {
    "mamba2_fp32_t64": dict(kind="mamba2", B=1, H=2, T=64, dk=16, dv=16, chunk=16, L=7,
                            io="f32", seed=0, shift=0.0),
    "mamba2_bf16_t2k": dict(kind="mamba2", B=2, H=8, T=2048, dk=64, dv=64, chunk=64, L=12,
                            io="bf16", seed=1, shift=2.0),
    "mamba2_bf16_t16k": dict(kind="mamba2", B=1, H=16, T=16384, dk=128, dv=128, chunk=64, L=15,
                             io="bf16", seed=2, shift=0.0),
    "gdn_bf16_t4k": dict(kind="gdn", B=2, H=16, T=4096, dk=128, dv=128, chunk=64, L=13,
                         io="bf16", seed=3, shift=2.0),
    # prefill continuation: 16384 new tokens at position 49152 (prefix held as
    # decode states, 17 slots), the long-context forward's distributions
    "mamba2_cont_bf16_t16k": dict(kind="mamba2_cont", B=1, H=16, T=16384, t0=49152, dk=128, dv=128, chunk=64,
                                  L=17, Ls=17, io="bf16", seed=2, shift=0.0),
    # the same workload under reading B (log-linear Mamba-2 on the delta-rule pseudo-values)
    "gdn_b_bf16_t4k": dict(kind="gdn_b", B=2, H=16, T=4096, dk=128, dv=128, chunk=64, L=13,
                           io="bf16", seed=3, shift=2.0),
    # backward of the long-context forward: its inputs plus an upstream gradient of o
    "mamba2_bwd_bf16_t16k": dict(kind="mamba2_bwd", B=1, H=16, T=16384, dk=128, dv=128, chunk=64, L=15,
                                 io="bf16", seed=2, shift=0.0),
    # one decay per level: the long-context forward's shape, log_alpha drawn
    # per token and level with the base distribution
    "level_decay_bf16_t16k": dict(kind="level_decay", B=1, H=16, T=16384, dk=128, dv=128, chunk=64, L=15,
                                  io="bf16", seed=6, shift=0.0),
    # prefix of 65536 tokens (forward with state export), then 256 decode steps
    "decode_b64_t64k": dict(kind="decode", B=64, H=32, T=65536, dk=128, dv=128, chunk=64, L=17,
                            Ls=17, steps=256, io="bf16", seed=4, shift=0.0),
    # Gated DeltaNet decode: the decode launch (64 x 32 heads, 17 level slots,
    # position 65536 on) with the Gated DeltaNet forward's distributions
    "gdn_decode_b64_t64k": dict(kind="gdn_decode", B=64, H=32, T=65536, dk=128, dv=128, chunk=64, L=17,
                                Ls=17, steps=256, io="bf16", seed=5, shift=2.0),
}

_MASK64 = (1 << 64) - 1


def _splitmix64(x: int) -> int:
    x = (x + 0x9E3779B97F4A7C15) & _MASK64
    x = ((x ^ (x >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    x = ((x ^ (x >> 27)) * 0x94D049BB133111EB) & _MASK64
    return x ^ (x >> 31)


def slice_seed(seed: int, name: str, b: int, h: int) -> int:
    """64-bit seed of one (tensor, b, h) slice; < 2**63 for torch."""
    x = _splitmix64(seed & _MASK64)
    for part in (zlib.crc32(name.encode()), b, h):
        x = _splitmix64(x ^ (part & _MASK64))
    return x & ((1 << 63) - 1)


def io_dtype(io: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[io]


def _normal(shape, seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def _uniform(shape, seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.rand(shape, generator=g, device=device, dtype=torch.float32)


def _fill(out, name, seed, draw, B, H, device, kind=None):
    """Fill out[b, h] with draw(kind, seed of (name, b, h)); `name` salts the
    seed, `kind` (default: name) selects the distribution."""
    for b in range(B):
        for h in range(H):
            out[b, h] = draw(kind or name, slice_seed(seed, name, b, h), device)


def make_inputs(cfg: dict, device="cpu", *, T=None, B=None, H=None, la_mode="softplus",
                lam_mode="softplus", lam_level=0, tag="", dout=None) -> dict:
    """Draw q, k, v, log_alpha, lam (and beta for Gated DeltaNet) for ``cfg``;
    with ``dout`` (default: for the backward workloads) also the upstream
    gradient dout [B,H,T,dv] in the io dtype.

    Shapes: q, k [B,H,T,dk]; v [B,H,T,dv] in the workload's io dtype;
    log_alpha [B,H,T], lam [B,H,T,L], beta [B,H,T] in float32.

    Kind "level_decay": log_alpha is [B,H,T,L], one draw per token and level.

    Parity-only variants: la_mode "zero" (alpha = 1) or "slow"
    (log_alpha ~ -U(0, 0.01)); lam_mode "const" (all lam = 1.5) or "onehot"
    (lam = 1 at level ``lam_level``, 0 elsewhere).  ``tag`` salts the seed.
    """
    B = cfg["B"] if B is None else B
    H = cfg["H"] if H is None else H
    T = cfg["T"] if T is None else T
    dk, dv, L = cfg["dk"], cfg["dv"], cfg["L"]
    seed = cfg["seed"] + (zlib.crc32(tag.encode()) << 8 if tag else 0)
    gdn = cfg["kind"] in ("gdn", "gdn_b")
    per_level = cfg["kind"] == "level_decay"
    dt = io_dtype(cfg["io"])
    shift = float(cfg.get("shift", 0.0))

    def draw(name, s, dev):
        if name == "q":
            return _normal((T, dk), s, dev) / math.sqrt(dk)
        if name == "k":
            x = _normal((T, dk), s, dev)
            if gdn:
                return x / x.norm(dim=-1, keepdim=True)
            return x / math.sqrt(dk)
        if name == "v":
            return _normal((T, dv), s, dev)
        if name == "log_alpha":
            shp = (T, L) if per_level else (T,)
            if la_mode == "zero":
                return torch.zeros(shp, device=dev)
            if la_mode == "slow":
                return -0.01 * _uniform(shp, s, dev)
            return -torch.nn.functional.softplus(_normal(shp, s, dev) + shift)
        if name == "lam":
            if lam_mode == "const":
                return torch.full((T, L), 1.5, device=dev)
            if lam_mode == "onehot":
                x = torch.zeros(T, L, device=dev)
                x[:, lam_level] = 1.0
                return x
            return torch.nn.functional.softplus(_normal((T, L), s, dev))
        if name == "beta":
            return torch.sigmoid(_normal((T,), s, dev))
        if name == "dout":
            return _normal((T, dv), s, dev)
        raise KeyError(name)

    out = {}
    shapes = {"q": (B, H, T, dk), "k": (B, H, T, dk), "v": (B, H, T, dv),
              "log_alpha": (B, H, T, L) if per_level else (B, H, T), "lam": (B, H, T, L)}
    if gdn:
        shapes["beta"] = (B, H, T)
    if dout if dout is not None else cfg["kind"] == "mamba2_bwd":
        shapes["dout"] = (B, H, T, dv)
    for name, shp in shapes.items():
        buf = torch.empty(shp, device=device, dtype=torch.float32)
        _fill(buf, name, seed, draw, B, H, device)
        out[name] = buf.to(dt) if name in ("q", "k", "v", "dout") else buf
    return out


def make_decode_inputs(cfg: dict, device="cpu", *, steps=None, B=None, H=None, per_level=False) -> dict:
    """Per-step decode inputs: q, k [S,B,H,dk], v [S,B,H,dv] (io dtype),
    log_alpha [S,B,H], lam [S,B,H,Ls+1] (float32); config-1 distributions.
    For kind "gdn_decode" also beta [S,B,H], with k L2-normalised,
    beta = sigmoid(N(0,1)) and log_alpha = -softplus(N(0,1) + shift).
    With ``per_level`` log_alpha is [S,B,H,Ls+1], one draw per level."""
    B = cfg["B"] if B is None else B
    H = cfg["H"] if H is None else H
    S = cfg["steps"] if steps is None else steps
    dk, dv, Ls = cfg["dk"], cfg["dv"], cfg["Ls"]
    seed = cfg["seed"] + 7919
    dt = io_dtype(cfg["io"])
    gdn = cfg["kind"] == "gdn_decode"
    shift = float(cfg.get("shift", 0.0)) if gdn else 0.0

    def draw(name, s, dev):
        if name == "q":
            return _normal((S, dk), s, dev) / math.sqrt(dk)
        if name == "k":
            x = _normal((S, dk), s, dev)
            if gdn:
                return x / x.norm(dim=-1, keepdim=True)
            return x / math.sqrt(dk)
        if name == "v":
            return _normal((S, dv), s, dev)
        if name == "log_alpha":
            return -torch.nn.functional.softplus(_normal((S, Ls + 1) if per_level else (S,), s, dev) + shift)
        if name == "lam":
            return torch.nn.functional.softplus(_normal((S, Ls + 1), s, dev))
        if name == "beta":
            return torch.sigmoid(_normal((S,), s, dev))
        raise KeyError(name)

    out = {}
    shapes = {"q": (B, H, S, dk), "k": (B, H, S, dk), "v": (B, H, S, dv),
              "log_alpha": (B, H, S, Ls + 1) if per_level else (B, H, S), "lam": (B, H, S, Ls + 1)}
    if gdn:
        shapes["beta"] = (B, H, S)
    for name, shp in shapes.items():
        buf = torch.empty(shp, device=device, dtype=torch.float32)
        _fill(buf, "dec_" + name, seed, draw, B, H, device, kind=name)
        # step-major layout [S, B, H, ...] so that one step is one contiguous slab
        buf = buf.movedim(2, 0).contiguous()
        out[name] = buf.to(dt) if name in ("q", "k", "v") else buf
    return out


def to_f64(x: torch.Tensor):
    """float64 NumPy copy of the values a tensor holds (bf16 upcast exactly)."""
    return x.detach().to("cpu").to(torch.float64).numpy()
