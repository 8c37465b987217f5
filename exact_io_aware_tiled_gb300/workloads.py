"""Seeded synthetic inputs for the attention workloads.

This module only draws random numbers and rounds them to the storage dtype;
it holds none of the attention arithmetic.  Tests, the benchmark and the
oracle-side checks all take their inputs from here, so both sides of a parity
comparison see bit-identical values.

Recipe (shapes follow the workloads the FlashAttention pages measure or
discuss: GPT-2-medium attention B=64, H=16, N=1024, d=64 and BERT-large at
N=512 -- agihunt.info summary of arXiv 2205.14135, results paragraph and
table; a 23,400-step day with 12 heads in fp16 -- marketmaker.cc,
introduction; butterfly block-sparse attention to 64K -- agihunt.info,
block-sparse paragraph):

* one ``numpy.random.Generator`` per tensor: ``default_rng([seed, stream])``
  with streams 0..3 for Q, K, V, dO;
* i.i.d. N(0, 1) drawn in float32, multiplied by ``input_scale``, then rounded
  to the storage dtype with round-to-nearest-even (torch CPU casts);
* key-padding lengths L_b = integers(lo, hi + 1) from stream 4;
* block-sparse: kept(I, J) iff I == J or I ^ J is a power of two over
  N / 128 blocks;
* grouped-query: K and V are drawn with ``H_kv`` heads ([B, H_kv, N, d]);
* the sliding window is a mask parameter (``window``) and draws nothing;
* outliers (FP8 error study): with ``outlier_rate`` > 0, tensor n (stream
  s) also draws, from ``default_rng([seed, 8 + s])``, a uniform mask and
  N(0, 1) values, and adds ``outlier_sd`` x value where mask < rate (before
  the dtype rounding): x = z + outlier_sd * o * Bernoulli(rate).  The pages
  give no input distribution for the FP8 comparison; this one puts rare
  coordinates an order of magnitude above the rest, the situation the
  pages say the rotation is for;
* the FP8 rotation's sign vector: ``rotation_signs`` draws d values of
  +-1 from ``default_rng([seed, 16])``.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional

import numpy as np
import torch

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def butterfly(nblocks: int) -> np.ndarray:
    i = np.arange(nblocks)[:, None]
    j = np.arange(nblocks)[None, :]
    x = i ^ j
    return ((x == 0) | ((x & (x - 1)) == 0)).astype(np.uint8)


@dataclass
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int = 64
    dtype: str = "bf16"
    causal: bool = False
    seqlen_range: Optional[tuple] = None      # (lo, hi) inclusive, or None
    sparse_butterfly: bool = False
    block_size: int = 128
    dropout_p: float = 0.0
    dropout_seed: int = 0x5EED
    dropout_offset: int = 0
    input_scale: float = 1.0
    seed: int = 20260
    seqlens: Optional[np.ndarray] = field(default=None, repr=False)
    block_mask: Optional[np.ndarray] = field(default=None, repr=False)
    H_kv: Optional[int] = None                # K/V heads (grouped-query); None -> H
    window: int = 0                           # causal sliding window of keys (0 = none)
    outlier_rate: float = 0.0                 # probability of an outlier entry
    outlier_sd: float = 0.0                   # outlier standard deviation

    def __post_init__(self):
        if self.seqlen_range is not None and self.seqlens is None:
            lo, hi = self.seqlen_range
            rng = np.random.default_rng([self.seed, 4])
            self.seqlens = rng.integers(lo, hi + 1, size=self.B).astype(np.int32)
        if self.sparse_butterfly and self.block_mask is None:
            nb = -(-self.N // self.block_size)
            self.block_mask = butterfly(nb)

    @property
    def torch_dtype(self):
        return DTYPES[self.dtype]

    @property
    def hkv(self) -> int:
        return self.H if self.H_kv is None else int(self.H_kv)

    def with_(self, **kw):
        return replace(self, **kw)


def _draw(shape, seed, stream, scale, dtype, outlier_rate=0.0, outlier_sd=0.0):
    rng = np.random.default_rng([seed, stream])
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if outlier_rate > 0.0:
        ro = np.random.default_rng([seed, 8 + stream])
        hit = ro.random(size=shape) < outlier_rate
        o = ro.standard_normal(size=shape, dtype=np.float32)
        x = x + np.where(hit, np.float32(outlier_sd) * o, np.float32(0.0))
    if scale != 1.0:
        x = x * np.float32(scale)
    return torch.from_numpy(x).to(DTYPES[dtype])


def rotation_signs(d: int, seed: int) -> np.ndarray:
    """d random signs (int8, +-1) for the FP8 path's rotation."""
    rng = np.random.default_rng([seed, 16])
    return (rng.integers(0, 2, size=d) * 2 - 1).astype(np.int8)


def make_inputs(wl: Workload, grads: bool = True):
    """q, do as [B,H,N,d] and k, v as [B,H_kv,N,d] torch CPU tensors of the storage dtype."""
    shp = (wl.B, wl.H, wl.N, wl.d)
    kshp = (wl.B, wl.hkv, wl.N, wl.d)
    out = {n: _draw(shp if n == "q" else kshp, wl.seed, s, wl.input_scale, wl.dtype,
                    wl.outlier_rate, wl.outlier_sd)
           for s, n in enumerate(("q", "k", "v"))}
    if grads:
        out["do"] = _draw(shp, wl.seed, 3, wl.input_scale, wl.dtype)
    return out


# The workloads (name -> Workload).  Seeds are 20260 + index.
CONFIGS = {
    "tiny_f32": Workload("tiny_f32", B=1, H=2, N=256, dtype="f32", seed=20261),
    "gpt2_medium_causal": Workload("gpt2_medium_causal", B=64, H=16, N=1024,
                                   dtype="bf16", causal=True, seed=20262),
    "bert_large_pad_dropout": Workload("bert_large_pad_dropout", B=32, H=16, N=512,
                                       dtype="bf16", seqlen_range=(256, 512),
                                       dropout_p=0.1, seed=20263),
    "long_ragged_causal_f16": Workload("long_ragged_causal_f16", B=1, H=12, N=23400,
                                       dtype="f16", causal=True, input_scale=0.5,
                                       seed=20264),
    "butterfly_sparse_64k": Workload("butterfly_sparse_64k", B=1, H=8, N=65536,
                                     dtype="bf16", sparse_butterfly=True, seed=20265),
    # grouped-query attention at the GPT-2-medium shape with 8 K/V heads
    # (living-dl-book, section 6: GQA-8)
    "gqa8_gpt2_medium_causal": Workload("gqa8_gpt2_medium_causal", B=64, H=16, N=1024, H_kv=8,
                                        dtype="bf16", causal=True, seed=20266),
    # the sliding-window exercise of lynx-cortex ("Problemas de práctica"):
    # N = 8192 with a window of 512 keys
    "window512_8k": Workload("window512_8k", B=4, H=16, N=8192, dtype="bf16", causal=True,
                             window=512, seed=20267),
    # head dimension 128 at the GPT-2-medium model width (8 heads x 128 =
    # 16 x 64), the case the pages single out as the one where the on-chip
    # tile budget gets tight (marketmaker.cc, "O que isso custou"; lynx-cortex,
    # "Lo que Flash forward no hace"); same FLOPs as the d = 64 workload
    "gpt2_medium_d128_causal": Workload("gpt2_medium_d128_causal", B=64, H=8, N=1024, d=128,
                                        dtype="bf16", causal=True, seed=20268),
    # FP8 forward (living-dl-book, section 10; marketmaker.cc, "FA3"): the
    # GPT-2-medium shape, bf16 inputs quantised to E4M3 per 128-row block
    # after the random rotation
    "gpt2_medium_causal_fp8": Workload("gpt2_medium_causal_fp8", B=64, H=16, N=1024, dtype="bf16",
                                       causal=True, seed=20269),
    # the FP8 forward at head dimension 128 (GPT-2-medium width: 8 heads of 128)
    "gpt2_medium_d128_causal_fp8": Workload("gpt2_medium_d128_causal_fp8", B=64, H=8, N=1024, d=128,
                                            dtype="bf16", causal=True, seed=20271),
    # FP8 error study: N(0, 1) plus 0.1 % outliers of standard deviation 10
    "outliers_fp8": Workload("outliers_fp8", B=1, H=4, N=2048, dtype="bf16", seed=20270,
                             outlier_rate=1e-3, outlier_sd=10.0),
}
