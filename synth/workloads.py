"""Synthetic workloads: parameter lists shaped like the pages' models.

Only parameter *shapes* matter to the shard-local step; no weights, tokens or
datasets are involved. Each list is in module-definition (registration) order,
with a tied entry naming the index of the parameter it shares storage with.
Values are drawn by ``synth`` (master ~ N(0, 0.02) fp32, gradients
~ N(0, 1e-3) bf16, seed 0).
"""
from __future__ import annotations

from dataclasses import dataclass, field


@dataclass(frozen=True)
class Param:
    name: str
    shape: tuple
    tied_to: int = -1

    @property
    def numel(self):
        n = 1
        for d in self.shape:
            n *= d
        return n


@dataclass(frozen=True)
class Workload:
    key: str
    title: str
    params: tuple
    world: int          # N, emulated data-parallel ranks
    stage: int          # ZeRO stage whose layout the config names (1, 2, 3)
    steps: int
    bucket_elems: int = 0
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01
    master_sigma: float = 0.02
    grad_sigma: float = 1e-3
    outlier_frac: float = 0.0
    outlier_scale: float = 1.0
    seed: int = 0
    align: int = 128
    notes: str = field(default="", compare=False)

    @property
    def numels(self):
        return [p.numel for p in self.params]

    @property
    def tied_to(self):
        return [p.tied_to for p in self.params]

    @property
    def hparams(self):
        return dict(lr=self.lr, beta1=self.beta1, beta2=self.beta2, eps=self.eps,
                    weight_decay=self.weight_decay)


def gpt2_params(n_layer, d, ffn, vocab, n_pos, tied=True):
    """GPT-2 layout: wte, [wpe], blocks of (ln_1, c_attn, attn c_proj, ln_2,
    c_fc, mlp c_proj) with biases, ln_f, [lm_head tied to wte]."""
    ps = [Param("wte", (vocab, d))]
    if n_pos:
        ps.append(Param("wpe", (n_pos, d)))
    for i in range(n_layer):
        h = f"h.{i}."
        ps += [
            Param(h + "ln_1.weight", (d,)), Param(h + "ln_1.bias", (d,)),
            Param(h + "attn.c_attn.weight", (d, 3 * d)), Param(h + "attn.c_attn.bias", (3 * d,)),
            Param(h + "attn.c_proj.weight", (d, d)), Param(h + "attn.c_proj.bias", (d,)),
            Param(h + "ln_2.weight", (d,)), Param(h + "ln_2.bias", (d,)),
            Param(h + "mlp.c_fc.weight", (d, ffn)), Param(h + "mlp.c_fc.bias", (ffn,)),
            Param(h + "mlp.c_proj.weight", (ffn, d)), Param(h + "mlp.c_proj.bias", (d,)),
        ]
    ps += [Param("ln_f.weight", (d,)), Param("ln_f.bias", (d,))]
    if tied:
        ps.append(Param("lm_head.weight", (vocab, d), tied_to=0))
    return tuple(ps)


def qwen2_params(n_layer, d, ffn, n_q, n_kv, head_dim, vocab, tied=True):
    """Qwen2 layout: embed, blocks of (input norm, q/k/v with bias, o without,
    post-attention norm, SwiGLU gate/up/down), final norm, [tied lm_head]."""
    q, kv = n_q * head_dim, n_kv * head_dim
    ps = [Param("embed_tokens", (vocab, d))]
    for i in range(n_layer):
        h = f"layers.{i}."
        ps += [
            Param(h + "input_layernorm", (d,)),
            Param(h + "q_proj.weight", (q, d)), Param(h + "q_proj.bias", (q,)),
            Param(h + "k_proj.weight", (kv, d)), Param(h + "k_proj.bias", (kv,)),
            Param(h + "v_proj.weight", (kv, d)), Param(h + "v_proj.bias", (kv,)),
            Param(h + "o_proj.weight", (d, q)),
            Param(h + "post_attention_layernorm", (d,)),
            Param(h + "gate_proj", (ffn, d)), Param(h + "up_proj", (ffn, d)),
            Param(h + "down_proj", (d, ffn)),
        ]
    ps.append(Param("norm", (d,)))
    if tied:
        ps.append(Param("lm_head", (vocab, d), tied_to=0))
    return tuple(ps)


def llama_params(n_layer, d, ffn, vocab):
    """Llama layout: embed, blocks of (input norm, q/k/v/o, post norm,
    gate/up/down), final norm, untied lm_head."""
    ps = [Param("embed_tokens", (vocab, d))]
    for i in range(n_layer):
        h = f"layers.{i}."
        ps += [
            Param(h + "input_layernorm", (d,)),
            Param(h + "q_proj", (d, d)), Param(h + "k_proj", (d, d)),
            Param(h + "v_proj", (d, d)), Param(h + "o_proj", (d, d)),
            Param(h + "post_attention_layernorm", (d,)),
            Param(h + "gate_proj", (ffn, d)), Param(h + "up_proj", (ffn, d)),
            Param(h + "down_proj", (d, ffn)),
        ]
    ps += [Param("norm", (d,)), Param("lm_head", (vocab, d))]
    return tuple(ps)


TINY = Workload(
    "tiny", "Tiny 2-layer transformer (d 256, FFN 1024, vocab 1000, tied), N=4, ZeRO-1",
    gpt2_params(2, 256, 1024, 1000, 0), world=4, stage=1, steps=3,
    notes="no position table; P = 1,836,032 with the stated dims")
GPT2_SMALL = Workload(
    "gpt2-small", "GPT-2-small (12 x d768, FFN 3072, vocab 50257, 1024 pos), N=8, ZeRO-2, "
    "25M-element buckets", gpt2_params(12, 768, 3072, 50257, 1024), world=8, stage=2,
    steps=10, bucket_elems=25_000_000)
QWEN25_3B = Workload(
    "qwen2.5-3b", "Qwen2.5-3B (36 x d2048, SwiGLU 11008, 16Q/2KV x 128, vocab 151936, tied), "
    "N=4, ZeRO-3 shard step", qwen2_params(36, 2048, 11008, 16, 2, 128, 151936), world=4,
    stage=3, steps=15)
LLAMA_7B = Workload(
    "llama-7b", "Llama-7B (32 x d4096, FFN 11008, vocab 32000), N=8, one rank's shard step, "
    "1% x100 gradient outliers", llama_params(32, 4096, 11008, 32000), world=8, stage=3,
    steps=10, outlier_frac=0.01, outlier_scale=100.0)

WORKLOADS = {w.key: w for w in (TINY, GPT2_SMALL, QWEN25_3B, LLAMA_7B)}

# The sweep: flat shard sizes x emulated ranks x incoming-gradient dtype x
# parameter dtype (2 = bf16, 3 = 3-byte, 4 = fp32).
SWEEP_SHARD_SIZES = [1 << k for k in range(10, 31, 2)]
SWEEP_WORLDS = [2, 4, 8, 16, 64]
SWEEP_GRAD_BYTES = [2, 4]
SWEEP_PARAM_BYTES = [2, 3, 4]


def wrap_units(w):
    """FSDP wrap units of a workload's parameter list: one unit per transformer
    block (the repeating architectural unit) and a root unit holding the rest
    (embeddings, final norm, head; a tied head stays with its embedding).
    Returns lists of indices into ``w.params``."""
    blocks, root = {}, []
    for i, p in enumerate(w.params):
        parts = p.name.split(".")
        if parts[0] in ("layers", "h") and len(parts) > 1 and parts[1].isdigit():
            blocks.setdefault(int(parts[1]), []).append(i)
        else:
            root.append(i)
    return [blocks[k] for k in sorted(blocks)] + [root]


def sweep_workload(S, world):
    """A one-tensor parameter list whose padded flat buffer is world*S."""
    return Workload(f"sweep-S{S}-N{world}", f"sweep shard {S} x N={world}",
                    (Param("flat", (world * S,)),), world=world, stage=3, steps=1)
