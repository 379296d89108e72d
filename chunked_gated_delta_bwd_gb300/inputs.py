"""Seeded synthetic inputs for the gated delta-rule backward.

This module draws random tensors and nothing else: it holds none of the
method's arithmetic, so both the CUDA path (tests, benchmark) and the oracle
can take their inputs from it.  Everything is generated on the CPU with one
``torch.Generator`` per case, in a fixed draw order:

    varlen lengths (if any), q, k, v, beta logits, gate inputs, h0, dht, dO

Value recipes (the workloads the pages benchmark):

* q, k, v, dO ~ N(0, 1), stored bf16 [T_total, H, D] (token-major);
* beta logits ~ N(0, 1), bf16 [T_total, H];
* GDN gate: g = -softplus(a), a ~ N(0, 1), float32 [T_total, H] (natural log);
* KDA gate inputs: g_raw ~ N(0, 1) bf16 [T_total, H, D], A_log ~ U(-1, 0) float32
  [H], dt_bias ~ N(0, 0.1) float32 [H, D]; the gate function is an API parameter
  carried along (``kda_gate``: "softplus", or "sigmoid" with ``gate_scale``; the pages
  print no value for gate_scale, the sigmoid cases use -2, a per-token decay of the
  same order as the softplus gate's);
* h0, dht ~ N(0, 0.1) float32 [N, H, D, D] where the case asks for them;
* varlen: N lengths ~ U[1, max_len] (integers), cu_seqlens int64 [N + 1].
"""
from dataclasses import dataclass, field
from typing import Optional

import torch


@dataclass(frozen=True)
class Case:
    name: str
    mode: str                 # "gdn" or "kda"
    num_seqs: int
    seq_len: int              # dense length (ignored when varlen)
    heads: int
    dim: int
    seed: int
    varlen_max: int = 0       # > 0: lengths ~ U[1, varlen_max]
    with_h0: bool = False
    with_dht: bool = False
    lengths: Optional[tuple] = None  # explicit lengths (overrides the dense / random ones)
    k_heads: Optional[int] = None     # q / k heads (GQA: fewer than `heads`, which counts v heads)
    kda_gate: str = "softplus"        # KDA gate function ("softplus" or "sigmoid")
    gate_scale: float = 0.0           # the sigmoid gate's scale
    note: str = field(default="", compare=False)


# The five benchmark workloads (sizes, seeds, distributions).
CASES = {
    "gdn_tiny": Case("gdn_tiny", "gdn", 1, 128, 2, 64, seed=0,
                     note="GDN bwd tiny: B=1 H=2 T=128 D=64, h0=0, no dht"),
    "gdn_b2_h16_t4k": Case("gdn_b2_h16_t4k", "gdn", 2, 4096, 16, 128, seed=1, with_h0=True,
                           with_dht=True, note="GDN bwd: B=2 H=16 T=4096 D=128, h0 and dht"),
    "kda_b1_h16_t8k": Case("kda_b1_h16_t8k", "kda", 1, 8192, 16, 128, seed=2,
                           note="KDA bwd: B=1 H=16 T=8192 D=128, h0=0, no dht"),
    "gdn_varlen_h32": Case("gdn_varlen_h32", "gdn", 16, 0, 32, 128, seed=3, varlen_max=4096,
                           note="GDN varlen bwd: 16 packed sequences, lengths U[1,4096], H=32"),
    "kda_sigmoid_b1_h16_t8k": Case("kda_sigmoid_b1_h16_t8k", "kda", 1, 8192, 16, 128, seed=5, with_h0=True,
                                   with_dht=True, kda_gate="sigmoid", gate_scale=-2.0,
                                   note="KDA with the sigmoid-bounded gate: B=1 H=16 T=8192 D=128"),
    "gdn_gqa_hk16_hv32_t4k": Case("gdn_gqa_hk16_hv32_t4k", "gdn", 1, 4096, 32, 128, seed=6, with_h0=True,
                                  with_dht=True, k_heads=16,
                                  note="GDN with grouped q/k heads: 16 q/k heads, 32 v heads, T=4096"),
    "gdn_h16_t32k": Case("gdn_h16_t32k", "gdn", 1, 32768, 16, 128, seed=4, with_h0=True,
                         with_dht=True, note="long-sequence GDN bwd: B=1 H=16 T=32768 D=128"),
    "kda_h16_t32k": Case("kda_h16_t32k", "kda", 1, 32768, 16, 128, seed=4, with_h0=True,
                         with_dht=True, note="long-sequence KDA bwd: B=1 H=16 T=32768 D=128"),
}


def lengths_of(case: Case, gen: torch.Generator):
    if case.lengths is not None:
        return [int(x) for x in case.lengths]
    if case.varlen_max > 0:
        return torch.randint(1, case.varlen_max + 1, (case.num_seqs,), generator=gen).tolist()
    return [case.seq_len] * case.num_seqs


def make(case: Case):
    """Returns a dict of CPU tensors for ``case`` (see the module docstring)."""
    gen = torch.Generator().manual_seed(case.seed)
    lens = lengths_of(case, gen)
    cu = torch.zeros(len(lens) + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0)
    T, H, D, N = int(cu[-1]), case.heads, case.dim, len(lens)

    def normal(*shape, std=1.0, dtype=torch.bfloat16):
        return (torch.randn(*shape, generator=gen) * std).to(dtype)

    x = {"cu_seqlens": cu, "scale": D ** -0.5, "mode": case.mode}
    Hk = H if case.k_heads is None else case.k_heads
    x["q"] = normal(T, Hk, D)
    x["k"] = normal(T, Hk, D)
    x["v"] = normal(T, H, D)
    x["beta_logit"] = normal(T, H)
    if case.mode == "gdn":
        a = torch.randn(T, H, generator=gen)
        x["g"] = (-torch.nn.functional.softplus(a)).to(torch.float32)
    else:
        x["g_raw"] = normal(T, H, D)
        x["A_log"] = (torch.rand(H, generator=gen) - 1.0).to(torch.float32)
        x["dt_bias"] = normal(H, D, std=0.1, dtype=torch.float32)
        x["kda_gate"], x["gate_scale"] = case.kda_gate, case.gate_scale
    x["h0"] = normal(N, H, D, D, std=0.1, dtype=torch.float32) if case.with_h0 else None
    x["dht"] = normal(N, H, D, D, std=0.1, dtype=torch.float32) if case.with_dht else None
    x["dO"] = normal(T, H, D)
    return x


def conv_case(lengths, channels, width, seed, with_bias=True, silu=True):
    """Inputs of the causal conv1d backward: x, dy ~ N(0, 1) bf16 [T_total, C] (token-major;
    in a GDN layer C = the q, k and v channels), weight ~ N(0, 0.25) float32 [C, K], bias ~
    N(0, 0.1) float32 [C] (or None), packed sequences of the given lengths."""
    gen = torch.Generator().manual_seed(seed)
    cu = torch.zeros(len(lengths) + 1, dtype=torch.int64)
    cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0)
    T = int(cu[-1])
    x = torch.randn(T, channels, generator=gen).to(torch.bfloat16)
    w = (torch.randn(channels, width, generator=gen) * 0.5).to(torch.float32)
    b = (torch.randn(channels, generator=gen) * 0.1).to(torch.float32) if with_bias else None
    dy = torch.randn(T, channels, generator=gen).to(torch.bfloat16)
    return {"cu_seqlens": cu, "x": x, "weight": w, "bias": b, "dy": dy, "silu": silu}


def custom(mode, lengths, heads, dim, seed, with_h0=False, with_dht=False, kda_gate="softplus", gate_scale=0.0,
           k_heads=None):
    """A case with explicit sequence lengths (ragged tails, empty sequences, ...)."""
    return make(Case("custom", mode, len(lengths), 0, heads, dim, seed, with_h0=with_h0,
                     with_dht=with_dht, lengths=tuple(lengths), kda_gate=kda_gate, gate_scale=gate_scale,
                     k_heads=k_heads))
