"""Seeded synthetic inputs: model shapes, random weights, KV caches, token ids.

This module holds none of the method's arithmetic. It only draws random
numbers, so that the CUDA path and the CPU oracle can be fed identical bytes.

Recipe (the pages print no weights or workloads beyond the model names, so all
inputs are synthetic):
  * matrices and the embedding: bf16(N(0, 0.02));
  * RMSNorm gains: bf16(1 + N(0, 0.02)) so the scale of activations is kept and
    the gain multiply is still exercised;
  * KV cache slots [0, ctx): bf16(N(0, 1)); slots past the context are zero;
  * token ids: uniform over the vocabulary.
Every draw comes from a ``torch.Generator`` seeded with the documented seed, in a
fixed order, on the device the caller names.
"""
from __future__ import annotations

import dataclasses

import torch


@dataclasses.dataclass(frozen=True)
class ModelShape:
    name: str
    n_layers: int
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    tied: bool
    rms_eps: float = 1e-5
    rope_theta: float = 10000.0

    def as_dict(self) -> dict:
        return dataclasses.asdict(self)

    def weight_bytes(self) -> int:
        H, D, F, V = self.hidden, self.head_dim, self.ffn, self.vocab
        per_layer = (H * (self.n_heads * D) * 2 + H * (self.n_kv_heads * D) * 2  # q, o ; k, v
                     + 3 * H * F + 2 * H)                                         # mlp + 2 gains
        total = self.n_layers * per_layer + H + V * H * (1 if self.tied else 2)
        return 2 * total


TINY = ModelShape("tiny", 2, 256, 4, 2, 64, 1024, 4096, tied=False, rope_theta=10000.0)
LLAMA_1B = ModelShape("llama-3.2-1b-shape", 16, 2048, 32, 8, 64, 8192, 128256, tied=True,
                      rope_theta=500000.0)
LLAMA_8B = ModelShape("llama-3.1-8b-shape", 32, 4096, 32, 8, 128, 14336, 128256, tied=False,
                      rope_theta=500000.0)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One decode workload: a model shape, a batch, context lengths and steps."""
    name: str
    shape: ModelShape
    batch: int
    ctx: tuple          # per-sequence context length before the first decode step
    steps: int
    capacity: int       # KV slots per sequence
    prompt: int = 0     # >0: the context is a prompt that is prefilled, not random KV
    weight_seed: int = 0
    kv_seed: int = 1
    token_seed: int = 2
    len_seed: int = 3


def _ragged_lengths(batch: int, lo: int, hi: int, seed: int) -> tuple:
    g = torch.Generator().manual_seed(seed)
    return tuple(int(v) for v in torch.randint(lo, hi + 1, (batch,), generator=g))


WORKLOADS = {
    "tiny": Workload("tiny", TINY, 1, (64,), 16, capacity=128, prompt=64),
    "llama1b": Workload("llama1b", LLAMA_1B, 1, (512,), 128, capacity=640),
    "llama1b_ctx8k": Workload("llama1b_ctx8k", LLAMA_1B, 1, (8192,), 64, capacity=8256),
    "llama8b": Workload("llama8b", LLAMA_8B, 1, (2048,), 64, capacity=2112),
    "llama1b_b8": Workload("llama1b_b8", LLAMA_1B, 8, _ragged_lengths(8, 128, 4096, 3), 64,
                           capacity=4160),
}


def _normal_bf16(shape, std, mean, gen, device):
    t = torch.empty(shape, dtype=torch.float32, device=device)
    t.normal_(mean=mean, std=std, generator=gen)
    return t.to(torch.bfloat16)


def make_weights(shape: ModelShape, seed: int = 0, device="cpu") -> dict:
    """Random-init weights in the nn.Linear layout ([out][in], bf16)."""
    dev = torch.device(device)
    g = torch.Generator(device=dev).manual_seed(seed)
    H, D, F, V = shape.hidden, shape.head_dim, shape.ffn, shape.vocab
    nh, nkv = shape.n_heads, shape.n_kv_heads
    w = {"embed": _normal_bf16((V, H), 0.02, 0.0, g, dev)}
    names = ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "wgate", "wup", "wdown")
    for n in names:
        w[n] = []
    for _ in range(shape.n_layers):
        w["attn_norm"].append(_normal_bf16((H,), 0.02, 1.0, g, dev))
        w["wq"].append(_normal_bf16((nh * D, H), 0.02, 0.0, g, dev))
        w["wk"].append(_normal_bf16((nkv * D, H), 0.02, 0.0, g, dev))
        w["wv"].append(_normal_bf16((nkv * D, H), 0.02, 0.0, g, dev))
        w["wo"].append(_normal_bf16((H, nh * D), 0.02, 0.0, g, dev))
        w["mlp_norm"].append(_normal_bf16((H,), 0.02, 1.0, g, dev))
        w["wgate"].append(_normal_bf16((F, H), 0.02, 0.0, g, dev))
        w["wup"].append(_normal_bf16((F, H), 0.02, 0.0, g, dev))
        w["wdown"].append(_normal_bf16((H, F), 0.02, 0.0, g, dev))
    w["final_norm"] = _normal_bf16((H,), 0.02, 1.0, g, dev)
    w["lm_head"] = None if shape.tied else _normal_bf16((V, H), 0.02, 0.0, g, dev)
    return w


def make_kv(shape: ModelShape, batch: int, capacity: int, ctx, seed: int = 1, device="cpu"):
    """Per-layer K and V caches [B][nkv][S][D] bf16: N(0,1) in [0, ctx_b), zero after."""
    dev = torch.device(device)
    g = torch.Generator(device=dev).manual_seed(seed)
    ks, vs = [], []
    shp = (batch, shape.n_kv_heads, capacity, shape.head_dim)
    for _ in range(shape.n_layers):
        for lst in (ks, vs):
            t = _normal_bf16(shp, 1.0, 0.0, g, dev)
            for b in range(batch):
                t[b, :, ctx[b]:, :] = 0
            lst.append(t)
    return ks, vs


def empty_kv(shape: ModelShape, batch: int, capacity: int, device="cpu"):
    shp = (batch, shape.n_kv_heads, capacity, shape.head_dim)
    ks = [torch.zeros(shp, dtype=torch.bfloat16, device=device) for _ in range(shape.n_layers)]
    vs = [torch.zeros(shp, dtype=torch.bfloat16, device=device) for _ in range(shape.n_layers)]
    return ks, vs


def make_tokens(vocab: int, count: int, seed: int = 2) -> torch.Tensor:
    g = torch.Generator().manual_seed(seed)
    return torch.randint(0, vocab, (count,), generator=g, dtype=torch.int64).to(torch.int32)


def step_tokens(wl: Workload) -> torch.Tensor:
    """Teacher-forced ids [steps][B] for the decode steps (never the model's argmax)."""
    return make_tokens(wl.shape.vocab, wl.steps * wl.batch, wl.token_seed + 100).view(
        wl.steps, wl.batch)


def prompt_tokens(wl: Workload) -> torch.Tensor:
    return make_tokens(wl.shape.vocab, wl.prompt, wl.token_seed)


def step_positions(wl: Workload, s: int) -> list:
    return [wl.ctx[b] + s for b in range(wl.batch)]


def bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 view of its bits (on the host)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view("uint16")


def oracle_weights(w: dict) -> dict:
    out = {}
    for k, v in w.items():
        if v is None:
            out[k] = None
        elif isinstance(v, list):
            out[k] = [bits(x) for x in v]
        else:
            out[k] = bits(v)
    return out
