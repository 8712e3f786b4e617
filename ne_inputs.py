"""Seeded synthetic inputs for causal grouped-query attention with rotary embeddings.

This module is shared by the CPU oracle, the tests and the benchmark.  It only
draws random tensors: it holds none of the attention arithmetic.

The workloads are the NanoEuler model shapes described on the pages
("NanoEuler: GPT-2 scale LLM in C and CUDA", model-configuration table:
small CPU model dim 128 with 4/2 heads at context 128; GPU pipeline dim 768
with 12/4 heads, 16 layers, context 512), plus a long-context stress shape.
There is no dataset: activations are iid N(0, 1) draws standing in for real
Q/K/V activations and upstream gradients of those shapes.

Recipe (identical for every workload): a CPU ``torch.Generator`` seeded with
the workload's seed draws fp32 N(0, 1) tensors in the order q, k, v, dO, all
laid out [B, T, H, d].  q and k are then multiplied by ``qk_scale``.  For the
stress shape, ``torch.randint`` on the same generator then draws one position
per (tensor, batch, head) for q, k and v, and that row is multiplied by 8.
Finally every tensor is rounded to bfloat16.  Multi-layer workloads use seed
``seed + layer`` for layer ``layer``.

Padded variable-length (SFT) workloads also draw one length per sequence
from a second CPU generator seeded with ``seed``: integers uniform on
[16, T], the same for every layer of the step.  The pages give no length
mix for their instruction data (pairs padded to the context); a uniform mix
keeps about half of the padded work and spans every tile count.
"""
from __future__ import annotations

import dataclasses

import torch

ROPE_THETA = 10000.0


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    Hq: int
    Hkv: int
    d: int
    seed: int
    qk_scale: float = 1.0
    outlier_rows: bool = False
    layers: int = 1
    theta: float = ROPE_THETA
    varlen: bool = False

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def pairs(self) -> int:
        """Causal (t, s) pairs per (batch, query head): s <= t."""
        return self.T * (self.T + 1) // 2

    def flops_fwd(self) -> float:
        """Algorithmic forward flops of one layer: QK^T and PV over causal pairs."""
        return 4.0 * self.d * self.pairs * self.B * self.Hq

    def flops_bwd(self) -> float:
        """Algorithmic backward flops of one layer: five pair-wise contractions."""
        return 10.0 * self.d * self.pairs * self.B * self.Hq

    def tokens(self) -> int:
        return self.B * self.T

    def seqlens(self) -> list[int]:
        """Per-sequence valid lengths of a padded variable-length workload."""
        if not self.varlen:
            return [self.T] * self.B
        g = torch.Generator(device="cpu").manual_seed(self.seed)
        return torch.randint(16, self.T + 1, (self.B,), generator=g).tolist()

    def valid_pairs(self) -> int:
        """Causal (t, s) pairs summed over the sequences' valid rows."""
        return sum(L * (L + 1) // 2 for L in self.seqlens())


WORKLOADS = {
    w.name: w
    for w in (
        # NanoEuler small (CPU) model shape, a single sequence.
        Workload("tiny_b1_t128_h4x2_d32", B=1, T=128, Hq=4, Hkv=2, d=32, seed=1001),
        # NanoEuler small model shape, a training batch.
        Workload("small_b16_t128_h4x2_d32", B=16, T=128, Hq=4, Hkv=2, d=32, seed=1002),
        # NanoEuler 116M GPU model, one attention layer; q and k scaled by 0.5.
        Workload("gpt116m_b16_t512_h12x4_d64", B=16, T=512, Hq=12, Hkv=4, d=64, seed=1003,
                 qk_scale=0.5),
        # NanoEuler 116M model, the attention of a full step: 16 layers of B=64.
        Workload("gpt116m_step_16x_b64_t512_h12x4_d64", B=64, T=512, Hq=12, Hkv=4, d=64,
                 seed=1004, layers=16),
        # Decode against a KV cache at the 116M shape: one new token per sequence
        # (its query is the last row of q), 512 cached positions, 16 layers
        # with their own caches.
        Workload("gpt116m_decode_16x_b64_tk512_h12x4_d64", B=64, T=512, Hq=12, Hkv=4, d=64,
                 seed=1006, layers=16),
        # NanoEuler 116M SFT step: 16 layers of B=64 sequences padded to 512,
        # each with its own valid length.
        Workload("gpt116m_sft_16x_b64_t512_h12x4_d64", B=64, T=512, Hq=12, Hkv=4, d=64,
                 seed=1007, layers=16, varlen=True),
        # Long-context stress shape with one 8x row per (tensor, batch, head).
        Workload("stress_b4_t4096_h16x4_d128", B=4, T=4096, Hq=16, Hkv=4, d=128, seed=1005,
                 outlier_rows=True),
    )
}

TINY = WORKLOADS["tiny_b1_t128_h4x2_d32"]
SMALL = WORKLOADS["small_b16_t128_h4x2_d32"]
LAYER_116M = WORKLOADS["gpt116m_b16_t512_h12x4_d64"]
STEP_116M = WORKLOADS["gpt116m_step_16x_b64_t512_h12x4_d64"]
STRESS = WORKLOADS["stress_b4_t4096_h16x4_d128"]
DECODE_116M = WORKLOADS["gpt116m_decode_16x_b64_tk512_h12x4_d64"]
SFT_116M = WORKLOADS["gpt116m_sft_16x_b64_t512_h12x4_d64"]


def make_inputs(w: Workload, layer: int = 0) -> dict[str, torch.Tensor]:
    """Draw q, k, v, dO for one layer of workload ``w`` as contiguous CPU bf16 tensors."""
    g = torch.Generator(device="cpu").manual_seed(w.seed + layer)
    q = torch.randn(w.B, w.T, w.Hq, w.d, generator=g, dtype=torch.float32)
    k = torch.randn(w.B, w.T, w.Hkv, w.d, generator=g, dtype=torch.float32)
    v = torch.randn(w.B, w.T, w.Hkv, w.d, generator=g, dtype=torch.float32)
    do = torch.randn(w.B, w.T, w.Hq, w.d, generator=g, dtype=torch.float32)
    if w.qk_scale != 1.0:
        q.mul_(w.qk_scale)
        k.mul_(w.qk_scale)
    if w.outlier_rows:
        for x in (q, k, v):
            pos = torch.randint(0, w.T, (w.B, x.shape[2]), generator=g)
            for b in range(w.B):
                for h in range(x.shape[2]):
                    x[b, pos[b, h], h, :] *= 8.0
    return {name: x.to(torch.bfloat16).contiguous()
            for name, x in (("q", q), ("k", k), ("v", v), ("do", do))}


# q and k scale of the GPU tests' edge-case shapes: the 116M layer's
# (gpt116m_b16_t512: q and k x 0.5).  Those cases cover shapes (ragged T,
# head dims, groups, windows, lengths); unit-scale precision is covered by the
# unit-scale workloads above.
CUSTOM_QK_SCALE = 0.5


def make_custom(B: int, T: int, Hq: int, Hkv: int, d: int, seed: int,
                scale: float = 1.0) -> dict[str, torch.Tensor]:
    """Draw an arbitrary-shape case with the same recipe (used for edge-case tests)."""
    w = Workload("custom", B=B, T=T, Hq=Hq, Hkv=Hkv, d=d, seed=seed, qk_scale=scale)
    return make_inputs(w)


def as_f64(x: torch.Tensor):
    """Widen a bf16 tensor to a float64 numpy array (exact)."""
    return x.to(torch.float64).numpy()
