"""Seeded synthetic inputs for the dynamic-sparse-attention step.

This module is shared by the tests, the benchmark and the smoke check, and
feeds both the CUDA library and the CPU oracle the very same bytes. It holds
none of the method's arithmetic: it draws random tensors, rounds them to the
storage dtypes, and (for an INT8 cache) quantises them the way the synthetic
workload recipe states. Nothing here scores, selects or attends.

Workloads (the five shapes the library is measured on; the names say what
they are):

* ``decode_4k``      batch 1, 1 query token, context 4,096, 8 query heads over
                      2 KV heads, BF16 Q/K/V, top_k 512.
* ``grouped_decode_32k``  batch 4, 8 query tokens each, context 32,768,
                      24 query heads over 2 KV heads, BF16 query, FP16 KV,
                      top_k 2,048.
* ``decode_128k``    batch 1, 1 query token, context 131,072 (64 chunks of
                      2,048 keys), 24/2 heads, BF16 query, FP16 KV, top_k
                      2,048; 1 % of the index keys get a +3 sigma bias.
* ``prefill_8k_on_32k``  batch 1, 8,192 new tokens after a 32,768-token past
                      (cache length 40,960), 24/2 heads, BF16 throughout,
                      top_k 2,048.
* ``decode_256k_int8``  batch 1, 8 query tokens, context 262,144 (128 chunks),
                      INT8 KV with a per-token per-head fp32 absmax scale,
                      BF16 query, top_k 2,048.

Every workload has 16 index heads of dim 64 (BF16 qI/kI ~ N(0,1), fp32 head
weights w ~ U(0,1)) and head dim 128; Q/K/V ~ N(0,1).

Positions: the cache holds ``T`` rows and the ``S`` new query tokens are its
last ``S`` rows, so query ``s`` sits at position ``T - S + s`` and sees keys
``0 .. T - S + s`` (causal, including itself).
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import torch

# storage dtypes by name
DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16, "int8": torch.int8,
          "fp32": torch.float32}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    q_len: int            # S: new query tokens per sequence
    total_len: int        # T: cache rows visible to the last query token
    num_q_heads: int
    num_kv_heads: int
    top_k: int
    q_dtype: str = "bf16"
    kv_dtype: str = "bf16"
    head_dim: int = 128
    idx_heads: int = 16
    idx_dim: int = 64
    bias_frac: float = 0.0   # fraction of index keys given a +3 sigma shift
    capacity: Optional[int] = None  # cache rows allocated (>= total_len)
    seed: int = 1000

    @property
    def cap(self) -> int:
        return self.capacity if self.capacity is not None else self.total_len

    @property
    def query_tokens(self) -> int:
        return self.batch * self.q_len


WORKLOADS: Dict[str, Workload] = {
    "decode_4k": Workload("decode_4k", 1, 1, 4096, 8, 2, 512,
                          "bf16", "bf16", seed=1001),
    "grouped_decode_32k": Workload("grouped_decode_32k", 4, 8, 32768, 24, 2,
                                   2048, "bf16", "fp16", seed=1002),
    "decode_128k": Workload("decode_128k", 1, 1, 131072, 24, 2, 2048,
                            "bf16", "fp16", bias_frac=0.01, seed=1003),
    "prefill_8k_on_32k": Workload("prefill_8k_on_32k", 1, 8192, 40960, 24, 2,
                                  2048, "bf16", "bf16", seed=1004),
    "decode_256k_int8": Workload("decode_256k_int8", 1, 8, 262144, 24, 2, 2048,
                                 "bf16", "int8", seed=1005),
}


def quantize_int8(x: torch.Tensor):
    """Absmax INT8 codes over the last dim: scale = max|x|/127, code =
    clamp(round-half-even(x/scale), -127, 127); an all-zero row gets scale 0
    and codes 0. Returns (codes int8, scale fp32 with the last dim dropped)."""
    x = x.to(torch.float32)
    amax = x.abs().amax(dim=-1)
    scale = amax / 127.0
    safe = torch.where(scale > 0, scale, torch.ones_like(scale))
    codes = torch.round(x / safe.unsqueeze(-1)).clamp_(-127, 127)
    codes = torch.where(scale.unsqueeze(-1) > 0, codes, torch.zeros_like(codes))
    return codes.to(torch.int8), scale.contiguous()


def make_inputs(wl: Workload, seed: Optional[int] = None) -> Dict[str, torch.Tensor]:
    """CPU tensors for one workload, drawn in a fixed order from one seeded
    generator: qI, w, kI, bias mask, q, K, V.

    Returns a dict with qI [B,S,HI,DI] bf16, w [B,S,HI] fp32, kI [B,cap,DI]
    bf16, q [B,S,Hq,D], k/v [B,cap,Hkv,D] in the workload's dtypes, k_scale /
    v_scale [B,cap,Hkv] fp32 (INT8 only, else None), total_len [B] int32.
    """
    g = torch.Generator().manual_seed(wl.seed if seed is None else seed)
    B, S, cap = wl.batch, wl.q_len, wl.cap
    qI = torch.randn(B, S, wl.idx_heads, wl.idx_dim, generator=g)
    w = torch.rand(B, S, wl.idx_heads, generator=g)
    kI = torch.randn(B, cap, wl.idx_dim, generator=g)
    if wl.bias_frac > 0:
        nb = int(wl.bias_frac * wl.total_len)
        for b in range(B):
            pos = torch.randperm(wl.total_len, generator=g)[:nb]
            kI[b, pos] += 3.0
    q = torch.randn(B, S, wl.num_q_heads, wl.head_dim, generator=g)
    k = torch.randn(B, cap, wl.num_kv_heads, wl.head_dim, generator=g)
    v = torch.randn(B, cap, wl.num_kv_heads, wl.head_dim, generator=g)
    out = {
        "qI": qI.to(torch.bfloat16).contiguous(),
        "w": w.contiguous(),
        "kI": kI.to(torch.bfloat16).contiguous(),
        "q": q.to(DTYPES[wl.q_dtype]).contiguous(),
        "total_len": torch.full((B,), wl.total_len, dtype=torch.int32),
        "k_scale": None,
        "v_scale": None,
    }
    if wl.kv_dtype == "int8":
        out["k"], out["k_scale"] = quantize_int8(k)
        out["v"], out["v_scale"] = quantize_int8(v)
    else:
        out["k"] = k.to(DTYPES[wl.kv_dtype]).contiguous()
        out["v"] = v.to(DTYPES[wl.kv_dtype]).contiguous()
    return out


def make_append_inputs(batch: int, q_len: int, num_kv_heads: int, capacity: int,
                       total_len, q_dtype: str, kv_dtype: str, seed: int = 0,
                       specials: bool = True) -> Dict[str, torch.Tensor]:
    """CPU tensors for a cache append: the new tokens and the caches they are
    written into, from one seeded generator.

    New K/V rows are N(0,1) times a per-row magnitude 10^U(-3,3); with
    ``specials`` a few rows are replaced by an all-zero row, a row with one
    non-zero element, and (BF16 new tokens only) a row holding 70000 and 1e-6.
    The caches are filled with random sentinel values (INT8: random codes and
    positive scales) so that rows the append must not touch are recognisable.
    Returns kI_new [B,S,64] bf16, k_new / v_new [B,S,Hkv,128] q_dtype, kI
    [B,cap,64] bf16, k / v [B,cap,Hkv,128] kv_dtype, k_scale / v_scale
    [B,cap,Hkv] fp32 or None, total_len [B] int32.
    """
    g = torch.Generator().manual_seed(seed)
    B, S, H, cap = batch, q_len, num_kv_heads, capacity
    T = [int(t) for t in (total_len if hasattr(total_len, "__len__") else [total_len] * B)]
    kI_new = torch.randn(B, S, 64, generator=g).to(torch.bfloat16)
    new = []
    for _ in range(2):
        x = torch.randn(B, S, H, 128, generator=g)
        mag = 10.0 ** (torch.rand(B, S, H, 1, generator=g) * 6 - 3)
        x = x * mag
        if specials and B * S * H >= 3:
            flat = x.view(-1, 128)
            flat[0].zero_()
            flat[1].zero_()
            flat[1, 77] = -0.375
            if q_dtype == "bf16":
                flat[2, 5] = 70000.0
                flat[2, 6] = 1e-6
        new.append(x.to(DTYPES[q_dtype]).contiguous())
    out = {"kI_new": kI_new.contiguous(), "k_new": new[0], "v_new": new[1],
           "kI": torch.randn(B, cap, 64, generator=g).to(torch.bfloat16).contiguous(),
           "total_len": torch.tensor(T, dtype=torch.int32), "k_scale": None, "v_scale": None}
    for name in ("k", "v"):
        if kv_dtype == "int8":
            out[name] = torch.randint(-127, 128, (B, cap, H, 128), generator=g,
                                      dtype=torch.int64).to(torch.int8)
            out[name + "_scale"] = torch.rand(B, cap, H, generator=g) + 0.5
        else:
            out[name] = torch.randn(B, cap, H, 128, generator=g).to(DTYPES[kv_dtype]).contiguous()
    return out


def make_rope_inputs(tokens: int, heads: int, head_dim: int, rotary_dim: int, max_pos: int,
                     x_dtype: str, cos_dtype: str, seed: int = 0, first_pos: int = 0,
                     base: float = 1.0e6) -> Dict[str, torch.Tensor]:
    """CPU tensors for RMSNorm + rotary embedding: x [N, H, D] ~ N(0,1) times
    a per-vector magnitude 10^U(-2,2), gamma [D] ~ U(0.5, 1.5), the standard
    rotary angle table theta[p, i] = p * base^(-2i / rotary_dim) as cos / sin
    caches [max_pos, rotary_dim / 2] (computed in float64, stored in
    cos_dtype), and consecutive positions first_pos .. first_pos + N - 1."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(tokens, heads, head_dim, generator=g, dtype=torch.float64)
    x = x * 10.0 ** (torch.rand(tokens, heads, 1, generator=g, dtype=torch.float64) * 4 - 2)
    gamma = (torch.rand(head_dim, generator=g) + 0.5).float()
    h = rotary_dim // 2
    out = {"x": x.to(DTYPES[x_dtype]).contiguous(), "gamma": gamma,
           "positions": torch.arange(first_pos, first_pos + tokens, dtype=torch.int32),
           "cos": None, "sin": None}
    if h > 0:
        inv = base ** (-2.0 * torch.arange(h, dtype=torch.float64) / rotary_dim)
        theta = torch.arange(max_pos, dtype=torch.float64)[:, None] * inv[None, :]
        out["cos"] = torch.cos(theta).to(DTYPES[cos_dtype]).contiguous()
        out["sin"] = torch.sin(theta).to(DTYPES[cos_dtype]).contiguous()
    return out


def small_workload(name="small", batch=2, q_len=3, total_len=1000, num_q_heads=8,
                   num_kv_heads=2, top_k=64, q_dtype="bf16", kv_dtype="bf16",
                   capacity=None, bias_frac=0.0, seed=7) -> Workload:
    """A reduced-size workload of the same structure, for parity tests that the
    oracle finishes in seconds."""
    return Workload(name, batch, q_len, total_len, num_q_heads, num_kv_heads,
                    top_k, q_dtype, kv_dtype, bias_frac=bias_frac,
                    capacity=capacity, seed=seed)


def to_f64(t: Optional[torch.Tensor]):
    """Exact float64 numpy copy of a CPU tensor (bf16/fp16/int8/fp32 values are
    all exactly representable in float64)."""
    if t is None:
        return None
    return t.detach().to("cpu").to(torch.float64).numpy()
