"""Synthetic, seeded workloads for the 4-bit AdamW step: shapes and inputs only.

This module holds none of the optimizer's arithmetic.  It describes the five
parameter sets the step is checked and measured on and draws their seeded
inputs (initial FP32 weights and per-step BF16 gradients) with torch's own
generators, on whichever device the caller names.  Tests feed the same drawn
inputs to the CUDA library and to the CPU oracle; bench.py uses it to build
the measured workload.

Model shapes follow the architectures of the "Rounding in Preconditioner
Space" listing page (Table 6: GPT-style 1.4B is 24 layers, d=2048, FFN 8192)
and the public Qwen3-0.6B / Llama-3-8B layouts; no dataset or trained weight is
involved.  Tensors are PyTorch [out, in] matrices and 1-D vectors.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

T_LM_HEAD = 0x1
T_FACTORED = 0x2

# Hyperparameters used by every workload (lr, betas, eps, weight decay).
HYPER = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1)


@dataclass(frozen=True)
class TensorSpec:
    name: str
    shape: tuple
    flags: int = 0

    @property
    def numel(self) -> int:
        return math.prod(self.shape)

    @property
    def rows(self) -> int:
        return self.shape[0] if len(self.shape) >= 2 else 1


@dataclass(frozen=True)
class Workload:
    name: str
    tensors: tuple
    recipe: str            # "zip_sr" | "ze_eden" | "factored"
    grad: str              # gradient recipe, see draw_grad
    first_step: int = 1
    lm_head_sr: bool = False
    sigma_range: tuple = (1e-3, 1e-3)
    zero_block_frac: float = 0.0

    @property
    def numel(self) -> int:
        return sum(t.numel for t in self.tensors)


def _gpt_1p4b():
    d, f, v, L = 2048, 8192, 50304, 24
    ts = [TensorSpec("wte", (v, d), T_LM_HEAD | T_FACTORED)]
    for i in range(L):
        p = f"h{i}."
        ts += [TensorSpec(p + "ln1.w", (d,)), TensorSpec(p + "ln1.b", (d,)),
               TensorSpec(p + "attn.qkv.w", (3 * d, d), T_FACTORED), TensorSpec(p + "attn.qkv.b", (3 * d,)),
               TensorSpec(p + "attn.proj.w", (d, d), T_FACTORED), TensorSpec(p + "attn.proj.b", (d,)),
               TensorSpec(p + "ln2.w", (d,)), TensorSpec(p + "ln2.b", (d,)),
               TensorSpec(p + "mlp.fc.w", (f, d), T_FACTORED), TensorSpec(p + "mlp.fc.b", (f,)),
               TensorSpec(p + "mlp.proj.w", (d, f), T_FACTORED), TensorSpec(p + "mlp.proj.b", (d,))]
    ts += [TensorSpec("ln_f.w", (d,)), TensorSpec("ln_f.b", (d,))]
    return tuple(ts)


def _qwen3_0p6b():
    d, f, v, L, hq, hkv, hd = 1024, 3072, 151936, 28, 16, 8, 128
    ts = [TensorSpec("embed", (v, d), T_LM_HEAD | T_FACTORED)]
    for i in range(L):
        p = f"l{i}."
        ts += [TensorSpec(p + "input_norm", (d,)),
               TensorSpec(p + "q_proj", (hq * hd, d), T_FACTORED),
               TensorSpec(p + "k_proj", (hkv * hd, d), T_FACTORED),
               TensorSpec(p + "v_proj", (hkv * hd, d), T_FACTORED),
               TensorSpec(p + "o_proj", (d, hq * hd), T_FACTORED),
               TensorSpec(p + "q_norm", (hd,)), TensorSpec(p + "k_norm", (hd,)),
               TensorSpec(p + "post_norm", (d,)),
               TensorSpec(p + "gate", (f, d), T_FACTORED), TensorSpec(p + "up", (f, d), T_FACTORED),
               TensorSpec(p + "down", (d, f), T_FACTORED)]
    ts += [TensorSpec("norm", (d,))]
    return tuple(ts)


def _llama_8b():
    d, f, v, L, hkv, hd = 4096, 14336, 128256, 32, 8, 128
    ts = [TensorSpec("embed", (v, d), T_FACTORED)]
    for i in range(L):
        p = f"l{i}."
        ts += [TensorSpec(p + "input_norm", (d,)),
               TensorSpec(p + "q_proj", (d, d), T_FACTORED),
               TensorSpec(p + "k_proj", (hkv * hd, d), T_FACTORED),
               TensorSpec(p + "v_proj", (hkv * hd, d), T_FACTORED),
               TensorSpec(p + "o_proj", (d, d), T_FACTORED),
               TensorSpec(p + "post_norm", (d,)),
               TensorSpec(p + "gate", (f, d), T_FACTORED), TensorSpec(p + "up", (f, d), T_FACTORED),
               TensorSpec(p + "down", (d, f), T_FACTORED)]
    ts += [TensorSpec("norm", (d,)), TensorSpec("lm_head", (v, d), T_LM_HEAD | T_FACTORED)]
    return tuple(ts)


WORKLOADS = {
    # 1-D 4096 vector, ZIP-SR, g ~ N(0, 1e-3) redrawn every step, 10 steps.
    "vec4096_zipsr": Workload("vec4096_zipsr", (TensorSpec("p", (4096,)),), "zip_sr", "normal"),
    # One 4096x4096 matrix, ZE-EDEN; g = N(0,1) * per-row log-uniform scale in
    # [1e-6, 1e-2], a fixed 5% of the 128-blocks exactly zero; 100 steps.
    "mat4096_zeeden": Workload("mat4096_zeeden", (TensorSpec("w", (4096, 4096)),), "ze_eden", "row_scaled",
                               sigma_range=(1e-6, 1e-2), zero_block_frac=0.05),
    # GPT-style 1.4B (tied head), ZIP-SR, LM-head SR active: steps 9001.. of 10k.
    "gpt1p4b_zipsr": Workload("gpt1p4b_zipsr", _gpt_1p4b(), "zip_sr", "tensor_scaled", first_step=9001,
                              lm_head_sr=True, sigma_range=(1e-5, 1e-2)),
    # Qwen3-0.6B-shaped list, factored v for rank >= 2, g ~ N(0, 1e-3).
    "qwen0p6b_factored": Workload("qwen0p6b_factored", _qwen3_0p6b(), "factored", "normal"),
    # Llama-style 8B, ZIP-SR and ZE-EDEN; per-tensor scale log-uniform [1e-6, 1e-2].
    "llama8b_zipsr": Workload("llama8b_zipsr", _llama_8b(), "zip_sr", "tensor_scaled", sigma_range=(1e-6, 1e-2)),
    "llama8b_zeeden": Workload("llama8b_zeeden", _llama_8b(), "ze_eden", "tensor_scaled",
                               sigma_range=(1e-6, 1e-2)),
    # The paper's TorchAO 4-bit baseline (SDyn4-RTN m, Lin4-NZ State-RTN v) on
    # the same parameter sets, for comparison.
    "llama8b_torchao": Workload("llama8b_torchao", _llama_8b(), "torchao", "tensor_scaled",
                                sigma_range=(1e-6, 1e-2)),
    "gpt1p4b_torchao": Workload("gpt1p4b_torchao", _gpt_1p4b(), "torchao", "tensor_scaled", first_step=9001,
                                lm_head_sr=True, sigma_range=(1e-5, 1e-2)),
}


def _gen(device, *key) -> torch.Generator:
    g = torch.Generator(device=device)
    h = 0x9E3779B97F4A7C15
    for k in key:
        h = (h ^ (int(k) + 0x632BE59BD9B9E01 + (h << 6) + (h >> 2))) & 0xFFFFFFFFFFFFFFFF
    g.manual_seed(h & 0x7FFFFFFFFFFFFFFF)
    return g


def tensor_sigma(w: Workload, tensor_id: int, seed: int = 0) -> float:
    """Per-tensor gradient scale: log-uniform in w.sigma_range (fixed per tensor)."""
    lo, hi = w.sigma_range
    if lo == hi:
        return lo
    u = torch.rand(1, generator=_gen("cpu", seed, 17, tensor_id), dtype=torch.float64).item()
    return math.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))


def init_param(spec: TensorSpec, tensor_id: int, device="cpu", seed: int = 0, std: float = 0.02,
               n: int | None = None) -> torch.Tensor:
    """FP32 master weights ~ N(0, std); n draws only that many leading elements."""
    g = _gen(device, seed, 1, tensor_id)
    return torch.randn(spec.numel if n is None else n, generator=g, device=device, dtype=torch.float32).mul_(std)


def zero_block_mask(w: Workload, spec: TensorSpec, tensor_id: int, device="cpu", seed: int = 0) -> torch.Tensor:
    """Boolean per-128-block mask of blocks whose gradient is exactly zero at every step."""
    nb = (spec.numel + 127) // 128
    if w.zero_block_frac <= 0:
        return torch.zeros(nb, dtype=torch.bool, device=device)
    g = _gen(device, seed, 4, tensor_id)
    return torch.rand(nb, generator=g, device=device) < w.zero_block_frac


def draw_grad(w: Workload, spec: TensorSpec, tensor_id: int, step: int, device="cpu", seed: int = 0,
              out: torch.Tensor | None = None, n: int | None = None) -> torch.Tensor:
    """BF16 gradient of tensor `tensor_id` at step `step` (flat, numel; n: only
    that many leading elements, drawn directly, for timing samples)."""
    if n is not None and n < spec.numel and (w.grad == "row_scaled" or w.zero_block_frac > 0):
        return draw_grad(w, spec, tensor_id, step, device, seed)[:n].contiguous()
    g = _gen(device, seed, 2, tensor_id, step)
    n = spec.numel if n is None else n
    x = torch.randn(n, generator=g, device=device, dtype=torch.float32)
    if w.grad == "normal":
        x.mul_(w.sigma_range[0])
    elif w.grad == "tensor_scaled":
        x.mul_(tensor_sigma(w, tensor_id, seed))
    elif w.grad == "row_scaled":
        rows = spec.rows
        gr = _gen(device, seed, 3, tensor_id)
        lo, hi = w.sigma_range
        u = torch.rand(rows, generator=gr, device=device, dtype=torch.float64)
        sig = torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo))).to(torch.float32)
        x.view(rows, -1).mul_(sig[:, None])
    else:
        raise ValueError(w.grad)
    if w.zero_block_frac > 0:
        mask = zero_block_mask(w, spec, tensor_id, device, seed)
        nb = mask.numel()
        pad = nb * 128 - n
        if pad:
            x = torch.cat([x, x.new_zeros(pad)])
        x.view(nb, 128)[mask] = 0
        x = x[:n]
    if out is None:
        return x.to(torch.bfloat16)
    out.copy_(x)
    return out


def custom(name: str, shapes, recipe: str, flags=None, grad="normal", sigma=(1e-3, 1e-3), first_step=1,
           lm_head_sr=False, zero_block_frac=0.0) -> Workload:
    """A small workload of arbitrary shapes (tests: ragged tails, odd block counts)."""
    flags = flags or [T_FACTORED if len(s) >= 2 else 0 for s in shapes]
    ts = tuple(TensorSpec(f"{name}{i}", tuple(s), f) for i, (s, f) in enumerate(zip(shapes, flags)))
    return Workload(name, ts, recipe, grad, first_step=first_step, lm_head_sr=lm_head_sr, sigma_range=sigma,
                    zero_block_frac=zero_block_frac)
