"""Seeded synthetic inputs shared by the tests, the bench and the CPU reference.

This module holds no arithmetic of the method: it only draws random tensors of the
right shapes and names the workload shapes.  Weights are N(0, 0.02^2), RMSNorm weights
1 + N(0, 0.02^2), activations N(0, 1), directly-fed modulation vectors N(0, 0.1^2),
sigma U(0.5, 1]; every tensor is rounded to bf16 so both sides see identical operands.
There are no trained weights, prompts or images: these stand in for them.

Weight layouts here are the logical ones ([out, in], MLP-in rows [gate; up]).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

WEIGHT_STD = 0.02
MOD_STD = 0.1


@dataclass(frozen=True)
class Widths:
    hidden: int
    heads: int
    head_dim: int
    mlp_hidden: int
    n_dual: int
    n_single: int
    in_channels: int = 128
    txt_dim: int = 7680
    time_dim: int = 256


KLEIN = Widths(hidden=3072, heads=24, head_dim=128, mlp_hidden=9216, n_dual=5, n_single=20)
TINY = Widths(hidden=256, heads=2, head_dim=128, mlp_hidden=768, n_dual=1, n_single=1)


@dataclass(frozen=True)
class Workload:
    """A shape: batch, text rows, target patch grid (rows, cols), reference grids."""
    name: str
    widths: Widths
    batch: int
    n_txt: int
    grid: tuple
    ref_grids: tuple = field(default_factory=tuple)

    @property
    def n_img(self) -> int:
        return self.grid[0] * self.grid[1]

    @property
    def n_ref(self) -> int:
        return sum(h * w for h, w in self.ref_grids)

    @property
    def n_tokens(self) -> int:
        return self.n_txt + self.n_img + self.n_ref


# The five workloads: tiny oracle case; one dual block and one single block at klein
# width over 512 text rows + a 64x64 grid; the full 1024x1024 step (128x128x32 latent,
# 2x2 patches -> 64x64 tokens); a 1920x1088 target (120 wide x 68 high patch grid) with
# one 1024x1024 reference, batch 4.
WORKLOADS = {
    "tiny": Workload("tiny", TINY, 1, 32, (8, 8)),
    "dual_block_1024": Workload("dual_block_1024", KLEIN, 1, 512, (64, 64)),
    "single_block_1024": Workload("single_block_1024", KLEIN, 1, 512, (64, 64)),
    "step_1024": Workload("step_1024", KLEIN, 1, 512, (64, 64)),
    "ref_1920x1088_b4": Workload("ref_1920x1088_b4", KLEIN, 4, 512, (68, 120), ((64, 64),)),
}


def generator(seed: int, device="cpu") -> torch.Generator:
    # a shape-only ("meta") request still needs a real generator object
    g = torch.Generator(device="cpu" if str(device) == "meta" else device)
    g.manual_seed(int(seed))
    return g


def normal(shape, std, gen, device="cpu", mean=0.0, draw_dtype=torch.float32) -> torch.Tensor:
    """N(mean, std^2) rounded to bf16.

    draw_dtype float64 (about 4x slower on the CPU) gives the same bf16 values on every host:
    torch's float32 CPU sampler rounds its transform differently on x86 and on Arm, which
    moves some values by one bf16 step; a float64 draw would have to land within about
    2^-44 of a bf16 rounding boundary for that to happen."""
    t = torch.randn(*shape, generator=gen, device=device, dtype=draw_dtype)
    return (t * std + mean).to(torch.bfloat16)


def mod_weights(wd: Widths, gen, device="cpu", draw_dtype=torch.float32, mod_std=WEIGHT_STD) -> dict:
    H = wd.hidden
    return {
        "t_in": normal((H, wd.time_dim), WEIGHT_STD, gen, device, draw_dtype=draw_dtype),
        "t_out": normal((H, H), WEIGHT_STD, gen, device, draw_dtype=draw_dtype),
        "mod": normal((17 * H, H), mod_std, gen, device, draw_dtype=draw_dtype),
    }


def stream_weights(wd: Widths, gen, device="cpu", draw_dtype=torch.float32, std=WEIGHT_STD) -> dict:
    H, F, D = wd.hidden, wd.mlp_hidden, wd.head_dim
    return {
        "qkv": normal((3 * H, H), std, gen, device, draw_dtype=draw_dtype),
        "q_norm": normal((D,), WEIGHT_STD, gen, device, mean=1.0, draw_dtype=draw_dtype),
        "k_norm": normal((D,), WEIGHT_STD, gen, device, mean=1.0, draw_dtype=draw_dtype),
        "out": normal((H, H), std, gen, device, draw_dtype=draw_dtype),
        "mlp_in": normal((2 * F, H), std, gen, device, draw_dtype=draw_dtype),
        "mlp_out": normal((H, F), std, gen, device, draw_dtype=draw_dtype),
    }


def single_weights(wd: Widths, gen, device="cpu", draw_dtype=torch.float32, std=WEIGHT_STD) -> dict:
    H, F, D = wd.hidden, wd.mlp_hidden, wd.head_dim
    return {
        "qkv_mlp": normal((3 * H + 2 * F, H), std, gen, device, draw_dtype=draw_dtype),
        "q_norm": normal((D,), WEIGHT_STD, gen, device, mean=1.0, draw_dtype=draw_dtype),
        "k_norm": normal((D,), WEIGHT_STD, gen, device, mean=1.0, draw_dtype=draw_dtype),
        "out": normal((H, H + F), std, gen, device, draw_dtype=draw_dtype),
    }


def model_weights(wd: Widths, seed: int, device="cpu", n_dual=None, n_single=None,
                  draw_dtype=torch.float32, block_std=WEIGHT_STD, mod_std=WEIGHT_STD) -> dict:
    """Every weight of the model, logical layouts, bf16.  block_std (the blocks' projection
    matrices) and mod_std (the 17H modulation projection) scale the same draws; the defaults
    are the recipe's 0.02."""
    g = generator(seed, device)
    H, C = wd.hidden, wd.in_channels
    w = {"mod": mod_weights(wd, g, device, draw_dtype=draw_dtype, mod_std=mod_std),
         "x_emb": normal((H, C), WEIGHT_STD, g, device, draw_dtype=draw_dtype),
         "ctx_emb": normal((H, wd.txt_dim), WEIGHT_STD, g, device, draw_dtype=draw_dtype),
         "proj_out": normal((C, H), WEIGHT_STD, g, device, draw_dtype=draw_dtype)}
    nd = wd.n_dual if n_dual is None else n_dual
    ns = wd.n_single if n_single is None else n_single
    w["dual"] = [(stream_weights(wd, g, device, draw_dtype=draw_dtype, std=block_std),
                  stream_weights(wd, g, device, draw_dtype=draw_dtype, std=block_std)) for _ in range(nd)]
    w["single"] = [single_weights(wd, g, device, draw_dtype=draw_dtype, std=block_std) for _ in range(ns)]
    return w


def step_inputs(wl: Workload, seed: int, device="cpu", draw_dtype=torch.float32) -> dict:
    """Activations of one step: latent tokens, reference tokens, text features, sigma."""
    g = generator(seed + 1000, device)
    wd = wl.widths
    out = {
        "img_tokens": normal((wl.batch, wl.n_img, wd.in_channels), 1.0, g, device, draw_dtype=draw_dtype),
        "ref_tokens": (normal((wl.batch, wl.n_ref, wd.in_channels), 1.0, g, device, draw_dtype=draw_dtype)
                       if wl.n_ref else None),
        "txt_emb": normal((wl.batch, wl.n_txt, wd.txt_dim), 1.0, g, device, draw_dtype=draw_dtype),
    }
    # reading R19: sigma_0 drawn from the seed in (0.5, 1]; one sigma per batch row
    s0 = 1.0 - 0.5 * torch.rand(1, generator=g, device=device, dtype=torch.float64).item()
    out["sigma"] = torch.full((wl.batch,), s0, dtype=torch.float32, device=device)
    return out


def block_inputs(wl: Workload, seed: int, device="cpu") -> dict:
    """Block-level inputs: the joint stream x [B, N, H] and a directly fed modulation
    vector [B, 17H] (N(0, 0.1^2))."""
    g = generator(seed + 2000, device)
    wd = wl.widths
    return {
        "x": normal((wl.batch, wl.n_tokens, wd.hidden), 1.0, g, device),
        "mod": normal((wl.batch, 17 * wd.hidden), MOD_STD, g, device),
    }
