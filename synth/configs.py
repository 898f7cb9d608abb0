"""Synthetic workload table for the ZeRO shard step.

Each workload fixes the parameter layout (a flat buffer of named tensors laid
end to end, as ZeRO's contiguous gradient buffer keeps them), the simulated
data-parallel degree N, the accumulation micro-steps G, the gradient dtype and
distribution, the optimizer hyper-parameters, the loss-scaler settings and the
schedule of injected non-finite gradients.

Sources for the shapes and knobs:
  * DeepSpeed Complete Guide (youngju.dev), §2 memory table: fp16 params and
    grads, fp32 master / momentum / variance.
  * same page, §4.1 ds_config.json and §4.2 fp16 settings: eps 1e-8, initial
    scale 2^initial_scale_power with power 16, loss_scale_window 1000,
    min_loss_scale 1.
  * same page, §2.2: reduce_bucket_size 2e8 elements.
Values the pages leave open (lr where unstated, betas, init sigma, hysteresis,
step counts, the index of each injection) are fixed here as plain readings.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

ALIGN_ELEMS = 64


def gpt2_tensors(n_layer: int, d: int, vocab: int, n_ctx: int, d_ff: int | None = None):
    """GPT-2 style decoder with learned positions, biases everywhere and a tied head."""
    d_ff = d_ff or 4 * d
    t = [("wte", vocab * d), ("wpe", n_ctx * d)]
    for i in range(n_layer):
        p = f"h{i}."
        t += [
            (p + "ln_1.w", d), (p + "ln_1.b", d),
            (p + "attn.c_attn.w", d * 3 * d), (p + "attn.c_attn.b", 3 * d),
            (p + "attn.c_proj.w", d * d), (p + "attn.c_proj.b", d),
            (p + "ln_2.w", d), (p + "ln_2.b", d),
            (p + "mlp.c_fc.w", d * d_ff), (p + "mlp.c_fc.b", d_ff),
            (p + "mlp.c_proj.w", d_ff * d), (p + "mlp.c_proj.b", d),
        ]
    t += [("ln_f.w", d), ("ln_f.b", d)]
    return t


def llama_tensors(n_layer: int, d: int, d_ff: int, vocab: int):
    """Llama style decoder: no biases, RMSNorm weights, untied output head."""
    t = [("embed_tokens", vocab * d)]
    for i in range(n_layer):
        p = f"layers.{i}."
        t += [
            (p + "q_proj", d * d), (p + "k_proj", d * d), (p + "v_proj", d * d),
            (p + "o_proj", d * d),
            (p + "gate_proj", d * d_ff), (p + "up_proj", d * d_ff), (p + "down_proj", d_ff * d),
            (p + "input_layernorm", d), (p + "post_attention_layernorm", d),
        ]
    t += [("norm", d), ("lm_head", vocab * d)]
    return t


@dataclass
class Injection:
    step: int      # 1-based optimizer step
    micro: int     # 1-based micro-step
    rank: int      # simulated rank
    index: int     # flat parameter index
    kind: str      # "inf" or "nan"


@dataclass
class Workload:
    name: str
    stream: int
    tensors: list
    n: int
    g: int
    dtype: str                  # "fp16" | "bf16"
    sigma: float
    scale0: float
    dynamic: bool
    window: int
    steps: int
    lr: float
    weight_decay: float
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    hysteresis: int = 1
    min_scale: float = 1.0
    master_sigma: float = 0.02
    seed: int = 0
    tail_fraction: float = 0.0
    low_sigma_tensors: list = field(default_factory=list)   # (name, sigma)
    bucket_elems: int = 200_000_000
    injections: list = field(default_factory=list)

    @property
    def psi(self) -> int:
        return int(sum(n for _, n in self.tensors))

    @property
    def dtype_code(self) -> int:
        return 0 if self.dtype == "fp16" else 1

    def tensor_ranges(self):
        out, off = [], 0
        for name, n in self.tensors:
            out.append((name, off, off + n))
            off += n
        return out

    def injections_at(self, step: int):
        return [j for j in self.injections if j.step == step]


def _low_sigma_pick(tensors, frac: float, sigma: float, seed: int = 0):
    k = math.ceil(frac * len(tensors))
    perm = np.random.default_rng(seed).permutation(len(tensors))[:k]
    return [(tensors[i][0], sigma) for i in sorted(perm)]


def _every(k: int, steps: int):
    return list(range(k, steps + 1, k))


def make_workloads():
    gpt2 = gpt2_tensors(12, 768, 50257, 1024)
    dec13 = gpt2_tensors(24, 2048, 50257, 2048, d_ff=8192)
    llama7 = llama_tensors(32, 4096, 11008, 32000)
    psi7 = sum(n for _, n in llama7)
    psi13 = sum(n for _, n in dec13)
    w = {}
    w["flat-1m-n2"] = Workload(
        name="flat-1m-n2", stream=1, tensors=[("flat", 1 << 20)], n=2, g=1, dtype="fp16",
        sigma=1e-3, scale0=2.0 ** 16, dynamic=True, window=1000, steps=10, lr=1e-4,
        weight_decay=0.0, injections=[Injection(5, 1, 1, 12345, "inf")])
    w["gpt2-small-n8"] = Workload(
        name="gpt2-small-n8", stream=2, tensors=gpt2, n=8, g=4, dtype="fp16", sigma=1e-4,
        scale0=2.0 ** 16, dynamic=True, window=1000, steps=10, lr=1e-4, weight_decay=0.01,
        low_sigma_tensors=_low_sigma_pick(gpt2, 0.01, 1e-7))
    w["decoder-1.3b-n16"] = Workload(
        name="decoder-1.3b-n16", stream=3, tensors=dec13, n=16, g=2, dtype="bf16", sigma=5e-5,
        scale0=1.0, dynamic=False, window=1000, steps=20, lr=3e-4, weight_decay=0.1,
        tail_fraction=0.01,
        injections=[Injection(s, 1, (s // 7) % 16, (7919 * s) % psi13, "nan")
                    for s in _every(7, 20)])
    w["llama7b-zero3-n64"] = Workload(
        name="llama7b-zero3-n64", stream=4, tensors=llama7, n=64, g=1, dtype="fp16",
        sigma=1e-4, scale0=2.0 ** 16, dynamic=True, window=1000, steps=50, lr=1e-4,
        weight_decay=0.0)
    w["llama7b-n1"] = Workload(
        name="llama7b-n1", stream=5, tensors=llama7, n=1, g=8, dtype="fp16", sigma=1e-4,
        scale0=2.0 ** 16, dynamic=True, window=100, steps=200, lr=1e-4, weight_decay=0.01,
        injections=[Injection(s, 1, 0, (7919 * s) % psi7, "inf") for s in _every(100, 200)])
    return w


WORKLOADS = make_workloads()
