"""Seeded generators for MoE-LoRA layer inputs.

Shapes and value distributions follow the workloads the pages describe: a
GPT-OSS-20B-like MoE layer served with multi-LoRA (rank 32, 8 adapters in
parallel; vllm.com.cn "MoE multi-LoRA", results section, Fig. 3 caption) and the
hidden 4096 / intermediate 11008 / r = 32 example of the same page's Fig. 1.
No public dataset or benchmark is involved; every tensor is drawn here.

Layouts (row-major, the reduction dimension innermost, as nn.Linear stores
weights):

    x             [T, H]        bf16   activations, ~N(0, 1)
    logits        [T, E]        fp32   router logits
    token_adapter [T]           int32  adapter id per token, -1 = base model only
    W1            [E, 2I, H]    bf16   gate_up weights; rows [0, I) gate, [I, 2I) up
    W2            [E, H, I]     bf16   down weights
    A1            [L, E, r, H]  bf16   gate_up LoRA A (stored transposed: r x h_in)
    B1            [L, E, 2I, r] bf16   gate_up LoRA B (stored transposed: h_out x r)
    A2            [L, E, r, I]  bf16   down LoRA A
    B2            [L, E, H, r]  bf16   down LoRA B

Every value is drawn in fp32 with numpy's PCG64 generator and rounded to bf16
(round to nearest even) by torch. Draw order is fixed: routing, adapters, x,
W1, W2, A1, B1, A2, B2; large tensors are drawn one leading index at a time
so that host memory stays bounded.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence, Union

import numpy as np
import torch

# The five workloads the layer is measured on. "std" of weights is 0.02.
WORKLOADS = [
    dict(name="tiny", T=8, H=256, I=512, E=4, k=2, L=2, r=8,
         routing="gaussian", adapters="tiny"),
    dict(name="gptoss20b_decode", T=64, H=2880, I=2880, E=32, k=4, L=8, r=32,
         routing="gaussian", adapters="round_robin_shuffled"),
    dict(name="gptoss20b_prefill", T=4096, H=2880, I=2880, E=32, k=4, L=16, r=16,
         routing="zipf1.0", adapters="one_per_request16"),
    dict(name="paper_example_4096_11008", T=512, H=4096, I=11008, E=8, k=2, L=32, r=64,
         routing="gaussian", adapters="mixed_lengths"),
    dict(name="many_adapter_stress", T=256, H=2048, I=768, E=128, k=8, L=128, r=32,
         routing="gaussian", adapters="zipf1.1"),
]


WORKLOAD_NAMES = [w["name"] for w in WORKLOADS]

# Measured beside the five: a dense model served with multi-LoRA, the degenerate MoE of one
# expert taken by every token (E = 1, k = 1), at the size of an 8B-class dense model's MLP
# (hidden 4096, intermediate 14336), 64 decode tokens over 8 adapters of rank 16. Workload j
# of this list is seeded with 2000 + j.
EXTRA_WORKLOADS = [
    dict(name="dense_4096_14336", T=64, H=4096, I=14336, E=1, k=1, L=8, r=16,
         routing="gaussian", adapters="round_robin_shuffled"),
]
ALL_WORKLOAD_NAMES = WORKLOAD_NAMES + [w["name"] for w in EXTRA_WORKLOADS]


def _config_and_seed(index_or_name: Union[int, str]):
    """A workload's configuration and default seed: 1000 + i for the i-th of the five,
    2000 + j for the j-th extra one."""
    if isinstance(index_or_name, int):
        return WORKLOADS[index_or_name], 1000 + index_or_name
    names = [c["name"] for c in WORKLOADS]
    if index_or_name in names:
        i = names.index(index_or_name)
        return WORKLOADS[i], 1000 + i
    extra = [c["name"] for c in EXTRA_WORKLOADS]
    j = extra.index(index_or_name)  # ValueError for an unknown name
    return EXTRA_WORKLOADS[j], 2000 + j


def workload_by_name(name: str) -> dict:
    for c in WORKLOADS + EXTRA_WORKLOADS:
        if c["name"] == name:
            return dict(c)
    raise KeyError(name)


@dataclasses.dataclass
class LayerInputs:
    T: int
    H: int
    I: int
    E: int
    k: int
    L: int
    r: int
    x: torch.Tensor
    logits: torch.Tensor
    token_adapter: torch.Tensor
    W1: torch.Tensor
    W2: torch.Tensor
    A1: Optional[torch.Tensor]
    B1: Optional[torch.Tensor]
    A2: Optional[torch.Tensor]
    B2: Optional[torch.Tensor]
    name: str = "custom"
    seed: int = 0

    @property
    def S(self) -> int:
        return self.T * self.k


def _bf16_normal(rng: np.random.Generator, shape: Sequence[int], std: float) -> torch.Tensor:
    """N(0, std^2) drawn in fp32, rounded to bf16; one leading index at a time."""
    shape = tuple(int(s) for s in shape)
    out = torch.empty(shape, dtype=torch.bfloat16)
    if out.numel() == 0:
        return out
    if len(shape) <= 2:
        a = rng.standard_normal(size=shape, dtype=np.float32)
        a *= np.float32(std)
        out.copy_(torch.from_numpy(a))
        return out
    flat = out.view(-1, *shape[-2:])
    for i in range(flat.shape[0]):
        a = rng.standard_normal(size=shape[-2:], dtype=np.float32)
        a *= np.float32(std)
        flat[i].copy_(torch.from_numpy(a))
    return out


def _routing_logits(rng: np.random.Generator, T: int, E: int, routing: str) -> torch.Tensor:
    if routing == "gaussian":
        lg = rng.standard_normal(size=(T, E), dtype=np.float32)
    elif routing.startswith("zipf"):
        # Expert popularity p_e ~ (e+1)^-s. Adding Gumbel(0,1) noise to log p_e
        # and taking the k largest draws k distinct experts without replacement
        # with probability proportional to p (the Gumbel-top-k construction).
        s = float(routing[4:])
        logp = -s * np.log(np.arange(1, E + 1, dtype=np.float64))
        logp -= np.log(np.exp(logp).sum())
        u = rng.random(size=(T, E))
        u = np.maximum(u, 1e-300)
        gumbel = -np.log(-np.log(u))
        lg = (logp[None, :] + gumbel).astype(np.float32)
    else:
        raise ValueError(f"unknown routing {routing!r}")
    return torch.from_numpy(np.ascontiguousarray(lg))


def _adapters(rng: np.random.Generator, T: int, L: int, mode) -> torch.Tensor:
    if isinstance(mode, (list, tuple, np.ndarray, torch.Tensor)):
        a = np.asarray(mode, dtype=np.int32)
        assert a.shape == (T,)
    elif mode == "tiny":
        assert T == 8 and L >= 2
        a = rng.permutation(np.array([0, 1, 0, 1, 0, 1, -1, -1], dtype=np.int32))
    elif mode == "round_robin_shuffled":
        # one token per request, each adapter serving exactly T/L requests
        a = rng.permutation(np.arange(T, dtype=np.int32) % L)
    elif mode == "one_per_request16":
        # 16 requests of T/16 consecutive tokens; request q uses adapter perm[q]
        nreq = 16
        assert T % nreq == 0 and L >= nreq
        perm = rng.permutation(L)[:nreq].astype(np.int32)
        a = np.repeat(perm, T // nreq)
    elif mode == "mixed_lengths":
        # 32 requests of 1..64 tokens summing to T: every request starts with one
        # token and the rest are dealt one at a time to a uniformly chosen request
        # that is still below 64. Requests, in a seeded random order, are marked
        # adapter-free until they hold at least 10% of the tokens; the others draw
        # an adapter uniformly from [0, L).
        nreq, cap = 32, 64
        assert nreq <= T <= nreq * cap
        lengths = np.ones(nreq, dtype=np.int64)
        for _ in range(T - nreq):
            open_ = np.flatnonzero(lengths < cap)
            lengths[open_[rng.integers(len(open_))]] += 1
        need = int(round(0.1 * T))
        free = np.zeros(nreq, dtype=bool)
        got = 0
        for q in rng.permutation(nreq):
            if got >= need:
                break
            free[q] = True
            got += int(lengths[q])
        req_adapter = np.full(nreq, -1, dtype=np.int32)
        for q in range(nreq):
            if not free[q]:
                req_adapter[q] = rng.integers(0, L)
        a = np.repeat(req_adapter, lengths)
    elif mode.startswith("zipf"):
        s = float(mode[4:])
        p = np.arange(1, L + 1, dtype=np.float64) ** (-s)
        p /= p.sum()
        a = rng.choice(L, size=T, p=p).astype(np.int32)
    elif mode == "uniform_with_none":
        a = rng.integers(-1, L, size=T).astype(np.int32)
    elif mode == "none":
        a = np.full(T, -1, dtype=np.int32)
    else:
        raise ValueError(f"unknown adapter mode {mode!r}")
    return torch.from_numpy(np.ascontiguousarray(a.astype(np.int32)))


def make_layer_inputs(T: int, H: int, I: int, E: int, k: int, L: int, r: int, seed: int,
                      routing: str = "gaussian",
                      adapters: Union[str, Sequence[int]] = "uniform_with_none",
                      weight_std: float = 0.02,
                      lora_std: Optional[float] = 0.02,
                      name: str = "custom") -> LayerInputs:
    """Draw one layer's inputs.

    ``lora_std=None`` gives the "amplified adapter" variant: A ~ N(0, 1/fan_in)
    and B ~ N(0, 1/r), so that the low-rank term is as large as the base term.
    ``L == 0`` draws no adapter weights (base MoE only).
    """
    rng = np.random.default_rng(seed)
    logits = _routing_logits(rng, T, E, routing)
    if L > 0:
        token_adapter = _adapters(rng, T, L, adapters)
    else:
        token_adapter = torch.full((T,), -1, dtype=torch.int32)
    x = _bf16_normal(rng, (T, H), 1.0)
    W1 = _bf16_normal(rng, (E, 2 * I, H), weight_std)
    W2 = _bf16_normal(rng, (E, H, I), weight_std)
    if L > 0:
        a1 = lora_std if lora_std is not None else H ** -0.5
        a2 = lora_std if lora_std is not None else I ** -0.5
        b = lora_std if lora_std is not None else r ** -0.5
        A1 = _bf16_normal(rng, (L, E, r, H), a1)
        B1 = _bf16_normal(rng, (L, E, 2 * I, r), b)
        A2 = _bf16_normal(rng, (L, E, r, I), a2)
        B2 = _bf16_normal(rng, (L, E, H, r), b)
    else:
        A1 = B1 = A2 = B2 = None
    return LayerInputs(T=T, H=H, I=I, E=E, k=k, L=L, r=r, x=x, logits=logits,
                       token_adapter=token_adapter, W1=W1, W2=W2, A1=A1, B1=B1,
                       A2=A2, B2=B2, name=name, seed=seed)


def make_workload_inputs(index_or_name: Union[int, str], seed: Optional[int] = None) -> LayerInputs:
    """Inputs of a named workload (one of the five, or an extra one); the i-th of the five
    is seeded with 1000 + i, the j-th extra one with 2000 + j."""
    c, s0 = _config_and_seed(index_or_name)
    return make_layer_inputs(c["T"], c["H"], c["I"], c["E"], c["k"], c["L"], c["r"],
                             seed=s0 if seed is None else seed,
                             routing=c["routing"], adapters=c["adapters"], name=c["name"])


def make_workload_routing(index_or_name: Union[int, str], seed: Optional[int] = None):
    """Only the router logits and adapter ids of a named workload.

    Same generator and draw order as :func:`make_workload_inputs`, stopped before
    the activations and weights, so the values equal that function's.
    """
    c, s0 = _config_and_seed(index_or_name)
    rng = np.random.default_rng(s0 if seed is None else seed)
    logits = _routing_logits(rng, c["T"], c["E"], c["routing"])
    token_adapter = _adapters(rng, c["T"], c["L"], c["adapters"])
    return logits, token_adapter, dict(c)
