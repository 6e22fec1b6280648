"""Seeded synthetic inputs for the Gated DeltaNet core.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic, so both the CUDA path (through the binding) and the CPU
oracle can consume the same tensors.

The five workloads follow the shapes and value distributions of the layer core
described by "mlex 0.1.2, src/models/gated_delta.rs" (``GatedDeltaNet::load`` /
``GatedDeltaNet::forward``) and by the ``gatedDeltaUpdate`` tensor table of
"mlx-bun 0.4.0 -> 1.0.0, package/src/model/qwen3-delta.ts":

* qkv (pre-conv)   bf16 N(0, 1)           [B, T, C], C = 2*Hk*Dk + Hv*Dv
* conv weight      bf16 N(0, 0.5**2)      [C, K]   (std 0.5)
* a, b             bf16 N(0, 1)           [B, T, Hv]
* A_log            f32  log U[1, 16]      [Hv]
* dt_bias          f32  N(0, 0.5**2)      [Hv]
* conv_state       bf16 N(0, 1) or zeros  [B, K-1, C]
* state            f32  N(0, 0.05**2) or zeros [B, Hv, Dv, Dk]
* mask             u8   right padding from lengths L_b ~ U{1024..16384}

All tensors are CPU torch tensors drawn from ``torch.Generator`` with a fixed
seed (1000 + workload index for the per-call tensors; a per-step seed for
decode steps), so every run and every consumer sees identical bits.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Dims:
    """Problem sizes (the fields of ``GatedDeltaConfig`` plus B and T)."""

    B: int
    T: int
    Hk: int
    Hv: int
    Dk: int
    Dv: int
    K: int = 4
    eps_qk: float = 1e-6

    @property
    def key_dim(self) -> int:
        return self.Hk * self.Dk

    @property
    def value_dim(self) -> int:
        return self.Hv * self.Dv

    @property
    def C(self) -> int:
        """conv_dim: q channels, then k channels, then v channels."""
        return 2 * self.key_dim + self.value_dim

    def with_(self, **kw) -> "Dims":
        return dataclasses.replace(self, **kw)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    index: int
    dims: Dims
    steps: int = 1               # decode: carried steps; prefill: 1
    conv_state: str = "zeros"    # "zeros" | "normal"
    state: str = "zeros"         # "zeros" | "normal"
    ragged: bool = False         # right-padded rows with lengths U{lo..hi}
    len_lo: int = 0
    len_hi: int = 0


WORKLOADS = {
    "tiny": Workload("tiny", 0, Dims(B=1, T=8, Hk=1, Hv=2, Dk=32, Dv=32, K=4)),
    "decode_b1": Workload("decode_b1", 1, Dims(B=1, T=1, Hk=16, Hv=32, Dk=128, Dv=128, K=4),
                          steps=1024, conv_state="normal", state="normal"),
    "decode_b128": Workload("decode_b128", 2, Dims(B=128, T=1, Hk=16, Hv=32, Dk=128, Dv=128, K=4),
                            steps=256, conv_state="normal", state="normal"),
    "prefill_t8192": Workload("prefill_t8192", 3, Dims(B=1, T=8192, Hk=16, Hv=32, Dk=128, Dv=128, K=4)),
    "prefill_ragged": Workload("prefill_ragged", 4, Dims(B=8, T=16384, Hk=16, Hv=64, Dk=128, Dv=128, K=4),
                               state="normal", ragged=True, len_lo=1024, len_hi=16384),
}


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def _normal_bf16(shape, std: float, g: torch.Generator) -> torch.Tensor:
    return (torch.randn(shape, generator=g, dtype=torch.float32) * std).to(torch.bfloat16)


def make_params(d: Dims, seed: int) -> dict:
    """Per-layer parameters: conv weight [C, K] bf16, A_log and dt_bias [Hv] f32."""
    g = _gen(seed)
    conv_w = _normal_bf16((d.C, d.K), 0.5, g)
    A_log = torch.log(torch.empty(d.Hv, dtype=torch.float32).uniform_(1.0, 16.0, generator=g))
    dt_bias = torch.randn(d.Hv, generator=g, dtype=torch.float32) * 0.5
    return {"conv_w": conv_w, "A_log": A_log, "dt_bias": dt_bias}


def make_activations(d: Dims, seed: int) -> dict:
    """Per-call activations: qkv [B, T, C], a and b [B, T, Hv], all bf16 N(0, 1)."""
    g = _gen(seed)
    qkv = _normal_bf16((d.B, d.T, d.C), 1.0, g)
    a = _normal_bf16((d.B, d.T, d.Hv), 1.0, g)
    b = _normal_bf16((d.B, d.T, d.Hv), 1.0, g)
    return {"qkv": qkv, "a": a, "b": b}


def make_gate_inputs(d: Dims, seed: int) -> dict:
    """Inputs of the RMSNormGated output: z [B, T, Hv, Dv] bf16 N(0, 1) (the
    in_proj_z output) and the norm weight [Dv] f32 U[0.5, 1.5]."""
    g = _gen(seed)
    z = _normal_bf16((d.B, d.T, d.Hv, d.Dv), 1.0, g)
    norm_w = torch.empty(d.Dv, dtype=torch.float32).uniform_(0.5, 1.5, generator=g)
    return {"z": z, "norm_w": norm_w}


def make_states(d: Dims, seed: int, conv_state: str, state: str) -> dict:
    g = _gen(seed)
    if conv_state == "normal":
        cs = _normal_bf16((d.B, d.K - 1, d.C), 1.0, g)
    else:
        cs = torch.zeros((d.B, d.K - 1, d.C), dtype=torch.bfloat16)
    if state == "normal":
        st = torch.randn((d.B, d.Hv, d.Dv, d.Dk), generator=g, dtype=torch.float32) * 0.05
    else:
        st = torch.zeros((d.B, d.Hv, d.Dv, d.Dk), dtype=torch.float32)
    return {"conv_state": cs, "state": st}


def make_lengths(B: int, lo: int, hi: int, seed: int) -> torch.Tensor:
    """Row lengths drawn uniformly from the integers lo..hi (inclusive)."""
    return torch.randint(lo, hi + 1, (B,), generator=_gen(seed), dtype=torch.int64)


def right_padded_mask(lengths: torch.Tensor, T: int) -> torch.Tensor:
    """u8 [B, T]: 1 on the first L_b steps of row b, 0 after."""
    t = torch.arange(T, dtype=torch.int64)[None, :]
    return (t < lengths[:, None]).to(torch.uint8)


def random_mask(B: int, T: int, p_valid: float, seed: int) -> torch.Tensor:
    g = _gen(seed)
    return (torch.rand((B, T), generator=g) < p_valid).to(torch.uint8)


def workload_lengths(w: Workload, dims: Optional[Dims] = None) -> torch.Tensor:
    """Row lengths of a ragged workload (valid prefix of each row)."""
    d = dims or w.dims
    return make_lengths(d.B, min(w.len_lo, d.T), min(w.len_hi, d.T), 1000 + w.index + 104729)


def workload_inputs(w: Workload, dims: Optional[Dims] = None) -> dict:
    """All per-call tensors of a workload (CPU). ``dims`` may shrink the workload
    (same distributions, other sizes) for parity tests."""
    d = dims or w.dims
    seed = 1000 + w.index
    out = {"dims": d}
    out.update(make_params(d, seed))
    out.update(make_activations(d, seed + 7919))
    out.update(make_states(d, seed + 15485863, w.conv_state, w.state))
    if w.ragged:
        lens = workload_lengths(w, d)
        out["lengths"] = lens
        out["mask"] = right_padded_mask(lens, d.T)
    else:
        out["mask"] = None
    return out


def decode_step_inputs(w: Workload, step: int, dims: Optional[Dims] = None) -> dict:
    """Fresh qkv [B, 1, C], a, b [B, 1, Hv] for one decode step."""
    d = dims or w.dims
    return make_activations(d, (1000 + w.index) * 100003 + step)


def bf16_bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 array of its bit patterns (no arithmetic)."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view("uint16")
