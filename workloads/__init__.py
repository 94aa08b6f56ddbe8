"""Seeded synthetic inputs for the row-wise reduce-then-rescale workloads.

This module holds only input generation: shapes, value distributions and
structure (shifted rows, spikes).  It contains none of the arithmetic of
RMSNorm or softmax, and both the fp64 oracle's tests and the CUDA path's
tests and benchmark draw their inputs from it.

Recipe (every workload): one ``torch.Generator`` seeded with ``seed``
(default 0) on the requested device; binary32 samples are drawn in the order
x, residual, gamma, then the structure (shifted rows, spike columns); the cast
to bfloat16 (round-to-nearest-even) comes last.  Shapes follow the Qwen2.5-7B
numbers the pages use (hidden 3584, 28 heads, vocabulary 152064, scored
context 2048).  Masks are structure: entries set to -inf after sampling
(causal: key j > query i; keep-K: all but K seeded columns per row).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

_DT = {"f32": torch.float32, "bf16": torch.bfloat16}
ELEM_BYTES = {"f32": 4, "bf16": 2}


@dataclass(frozen=True)
class Workload:
    name: str
    op: str                 # "rmsnorm" | "fused_add_rmsnorm" | "layernorm" | "softmax" | "log_softmax" | "logsumexp" | "topk"
    M: int
    N: int                  # row length (H for the norms)
    in_dtype: str
    out_dtype: str
    sigma: float = 1.0      # std of the normal samples
    eps: float = 1e-6
    shift_rows: int = 0     # rows that get +shift added (softmax overflow check)
    low: float | None = None    # LayerNorm: x ~ U(low, high) instead of N(0, sigma^2)
    high: float | None = None
    shift: float = 1000.0
    spikes_per_row: int = 0
    spike: float = 30.0
    mask: str = ""          # "" | "causal" (square per head: query = row % N) | "keep:K"
    k: int = 0              # top-k: entries selected per row
    l2_resident: bool = False
    note: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def min_bytes(self) -> int:
        """Minimum HBM traffic of one call: each input read once, each output
        written once, gamma counted once."""
        e_in, e_out = ELEM_BYTES[self.in_dtype], ELEM_BYTES[self.out_dtype]
        n = self.M * self.N
        if self.op == "rmsnorm":
            return n * e_in + n * e_out + self.N * e_in
        if self.op == "layernorm":
            return n * e_in + n * e_out + 2 * self.N * e_in
        if self.op == "fused_add_rmsnorm":
            return 2 * n * e_in + 2 * n * e_out + self.N * e_in
        if self.op == "logsumexp":  # reads the rows, writes a float and an int64 per row
            return n * e_in + self.M * (4 + 8)
        if self.op == "topk":  # reads the rows; per row k values, indices and probs, one lse
            return n * e_in + self.M * self.k * (4 + 8 + 4) + self.M * 4
        return n * e_in + n * e_out


SWEEP_N = (32, 128, 1024, 4096, 32768, 152064)

WORKLOADS = {
    "rmsnorm_f32_64x3584": Workload(
        "rmsnorm_f32_64x3584", "rmsnorm", 64, 3584, "f32", "f32", sigma=1.0,
        l2_resident=True, note="RMSNorm fp32, 64 rows x hidden 3584"),
    "fused_add_rmsnorm_bf16_8192x4096": Workload(
        "fused_add_rmsnorm_bf16_8192x4096", "fused_add_rmsnorm", 8192, 4096, "bf16", "bf16",
        sigma=1.0, note="fused residual-add + RMSNorm bf16, batch 4 x seq 2048 x hidden 4096"),
    "softmax_attn_f32_114688x4096": Workload(
        "softmax_attn_f32_114688x4096", "softmax", 28 * 4096, 4096, "f32", "f32", sigma=3.0,
        shift_rows=round(0.01 * 28 * 4096),
        note="attention-score softmax fp32, 28 heads x 4096 queries x 4096 keys, 1% rows +1000"),
    "softmax_vocab_bf16_f32_64x152064": Workload(
        "softmax_vocab_bf16_f32_64x152064", "softmax", 64, 152064, "bf16", "f32", sigma=4.0,
        spikes_per_row=8, l2_resident=True,
        note="vocabulary-logit softmax, bf16 in / fp32 out, 64 rows x 152064, 8 spikes +30 per row"),
}
WORKLOADS["layernorm_f32_256x5120_mean101"] = Workload(
    "layernorm_f32_256x5120_mean101", "layernorm", 256, 5120, "f32", "f32", eps=1e-5,
    low=100.0, high=102.0, l2_resident=True,
    note="LayerNorm fp32, 256 x 5120, x ~ U(100, 102): mean >> std stress case")
WORKLOADS["layernorm_bf16_8192x4096"] = Workload(
    "layernorm_bf16_8192x4096", "layernorm", 8192, 4096, "bf16", "bf16", eps=1e-5, sigma=1.0,
    note="LayerNorm bf16, 8192 x 4096")
WORKLOADS["log_softmax_vocab_bf16_f32_64x152064"] = Workload(
    "log_softmax_vocab_bf16_f32_64x152064", "log_softmax", 64, 152064, "bf16", "f32", sigma=4.0,
    spikes_per_row=8, l2_resident=True,
    note="log-softmax of the vocabulary-logit rows, bf16 in / fp32 out")
WORKLOADS["logsumexp_argmax_vocab_bf16_64x152064"] = Workload(
    "logsumexp_argmax_vocab_bf16_64x152064", "logsumexp", 64, 152064, "bf16", "f32", sigma=4.0,
    spikes_per_row=8, l2_resident=True,
    note="sampling statistics of the vocabulary-logit rows: log-sum-exp and argmax, no probabilities")
WORKLOADS["logsumexp_argmax_vocab_bf16_1024x152064"] = Workload(
    "logsumexp_argmax_vocab_bf16_1024x152064", "logsumexp", 1024, 152064, "bf16", "f32", sigma=4.0,
    spikes_per_row=8,
    note="sampling statistics of a 1024-row batch of vocabulary-logit rows (311 MB)")
WORKLOADS["logsumexp_attn_bf16_114688x4096"] = Workload(
    "logsumexp_attn_bf16_114688x4096", "logsumexp", 28 * 4096, 4096, "bf16", "f32", sigma=3.0,
    shift_rows=round(0.01 * 28 * 4096),
    note="per-query log-sum-exp of bf16 attention scores, 28 heads x 4096 x 4096, 1% rows +1000")
WORKLOADS["topk_vocab_bf16_64x152064_k50"] = Workload(
    "topk_vocab_bf16_64x152064_k50", "topk", 64, 152064, "bf16", "f32", sigma=4.0,
    spikes_per_row=8, l2_resident=True, k=50,
    note="top-k sampling prologue of the vocabulary-logit rows: the 50 largest logits, "
         "their indices, their softmax and the row log-sum-exp")
WORKLOADS["softmax_causal_f32_57344x2048"] = Workload(
    "softmax_causal_f32_57344x2048", "softmax", 28 * 2048, 2048, "f32", "f32", sigma=3.0,
    mask="causal",
    note="causally masked attention-score softmax fp32, 28 heads x 2048 queries x 2048 keys: "
         "key j > query i is -inf (half the entries)")
WORKLOADS["softmax_topk_masked_bf16_f32_64x152064"] = Workload(
    "softmax_topk_masked_bf16_f32_64x152064", "softmax", 64, 152064, "bf16", "f32", sigma=4.0,
    mask="keep:64", l2_resident=True,
    note="vocabulary rows after a top-k style filter: all but 64 seeded columns per row are -inf")
WORKLOADS["softmax_attn_bf16_114688x4096"] = Workload(
    "softmax_attn_bf16_114688x4096", "softmax", 28 * 4096, 4096, "bf16", "bf16", sigma=3.0,
    shift_rows=round(0.01 * 28 * 4096),
    note="attention-score softmax with bf16 output, 28 heads x 4096 x 4096, 1% rows +1000")
# the pages' shape sweep: decode batch 1 and 32, a 2048-token prefill, a 16384-row batch
SHAPE_SWEEP_M = (1, 32, 2048, 16384)
for _m in SHAPE_SWEEP_M:
    _name = f"shape_rmsnorm_f32_{_m}x3584"
    WORKLOADS[_name] = Workload(_name, "rmsnorm", _m, 3584, "f32", "f32", sigma=1.0,
                                l2_resident=_m * 3584 * 8 < (64 << 20),
                                note=f"RMSNorm fp32 shape sweep, M={_m}, hidden 3584")
for _m in SHAPE_SWEEP_M:
    _name = f"shape_softmax_f32_{_m}x2048"
    WORKLOADS[_name] = Workload(_name, "softmax", _m, 2048, "f32", "f32", sigma=3.0,
                                l2_resident=_m * 2048 * 8 < (64 << 20),
                                note=f"score softmax fp32 shape sweep, M={_m}, context 2048")
for _n in SWEEP_N:
    _name = f"softmax_sweep_f32_N{_n}"
    WORKLOADS[_name] = Workload(_name, "softmax", (1 << 26) // _n, _n, "f32", "f32", sigma=2.0,
                                note=f"softmax fp32 sweep, 256 MiB per tensor, N={_n}")


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def rmsnorm_inputs(M, H, dtype="f32", sigma=1.0, fused=False, seed=0, device="cpu"):
    """x (and residual) ~ N(0, sigma^2), gamma ~ U(0.5, 1.5)."""
    g = _gen(device, seed)
    x = torch.randn(M, H, generator=g, device=device, dtype=torch.float32) * sigma
    res = None
    if fused:
        res = torch.randn(M, H, generator=g, device=device, dtype=torch.float32) * sigma
    gamma = torch.rand(H, generator=g, device=device, dtype=torch.float32) + 0.5
    out = {"x": x.to(_DT[dtype]), "gamma": gamma.to(_DT[dtype])}
    if fused:
        out["residual"] = res.to(_DT[dtype])
    return out


def layernorm_inputs(M, H, dtype="f32", sigma=1.0, low=None, high=None, seed=0, device="cpu"):
    """x ~ N(0, sigma^2) or U(low, high); gamma ~ U(0.5, 1.5); beta ~ N(0, 1)."""
    g = _gen(device, seed)
    if low is None:
        x = torch.randn(M, H, generator=g, device=device, dtype=torch.float32) * sigma
    else:
        x = torch.rand(M, H, generator=g, device=device, dtype=torch.float32) * (high - low) + low
    gamma = torch.rand(H, generator=g, device=device, dtype=torch.float32) + 0.5
    beta = torch.randn(H, generator=g, device=device, dtype=torch.float32)
    return {"x": x.to(_DT[dtype]), "gamma": gamma.to(_DT[dtype]), "beta": beta.to(_DT[dtype])}


def softmax_inputs(M, N, dtype="f32", sigma=1.0, shift_rows=0, shift=1000.0,
                   spikes_per_row=0, spike=30.0, seed=0, device="cpu", mask=""):
    """x ~ N(0, sigma^2); `shift_rows` distinct rows (seeded permutation) get
    +shift; each row gets `spikes_per_row` distinct seeded columns +spike;
    then `mask` sets entries to -inf: "causal" masks key j > query i, the
    query of row r being r mod N (square score blocks per head); "keep:K"
    keeps K distinct seeded columns of each row and masks the rest."""
    g = _gen(device, seed)
    x = torch.randn(M, N, generator=g, device=device, dtype=torch.float32) * sigma
    if shift_rows:
        rows = torch.randperm(M, generator=g, device=device)[:shift_rows]
        x[rows] += shift
    if spikes_per_row:
        for r in range(M):
            cols = torch.randperm(N, generator=g, device=device)[:spikes_per_row]
            x[r, cols] += spike
    if mask == "causal":
        q = (torch.arange(M, device=device) % N).unsqueeze(1)
        x.masked_fill_(torch.arange(N, device=device).unsqueeze(0) > q, float("-inf"))
    elif mask.startswith("keep:"):
        k = int(mask.split(":")[1])
        keep = torch.rand(M, N, generator=g, device=device).argsort(dim=1)[:, :k]
        masked = torch.full_like(x, float("-inf"))
        masked.scatter_(1, keep, x.gather(1, keep))
        x = masked
    elif mask:
        raise ValueError(f"unknown mask {mask!r}")
    return {"x": x.to(_DT[dtype])}


def make(w: Workload | str, seed=0, device="cpu"):
    """Inputs of a named workload, as torch tensors on `device`."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    if w.op == "layernorm":
        return layernorm_inputs(w.M, w.N, w.in_dtype, w.sigma, w.low, w.high, seed, device)
    if w.op in ("rmsnorm", "fused_add_rmsnorm"):
        return rmsnorm_inputs(w.M, w.N, w.in_dtype, w.sigma, w.op == "fused_add_rmsnorm",
                              seed, device)
    return softmax_inputs(w.M, w.N, w.in_dtype, w.sigma, w.shift_rows, w.shift,
                          w.spikes_per_row, w.spike, seed, device, w.mask)
