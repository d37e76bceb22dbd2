"""Seeded synthetic inputs for the GPTQ W4A16 linear layer.

This module is shared by the tests, the benchmark and the smoke check.  It
holds no arithmetic of the method (no unpacking, dequantization or product):
it only draws random tensors with the shapes and distributions of the
workloads below.

Packed words are drawn as uniformly random 32-bit patterns.  Every nibble of
such a word is then an independent uniform draw from 0..15, which is exactly
"q uniform on 0..15, packed eight to a word" without needing a packer here.

Workloads (Llama-7B and Llama-70B projection shapes stand in for real layers;
no checkpoint or dataset is used):

  single_layer   M=1, K=N=1024, g=128, trivial g_idx, no bias
  decode_7b      M in {1,2,4,8} x (K,N) in {(4096,4096), (4096,11008),
                 (11008,4096), (4096,12288)}, g=128, trivial, bias N(0, 0.1)
  actorder_7b    M in {1,4,16} x {(4096,11008), (11008,4096)}, g=128,
                 g_idx[k] = perm[k] // 128 for a seeded permutation
  prefill_7b     M in {512,2048} x {(4096,4096), (4096,11008), (11008,4096)},
                 g=128, trivial and act-order
  sweep_70b      (K,N) in {(8192,28672), (28672,8192), (8192,10240)} x
                 M in {1,2,4,8,16,32,64,128,256,2048} x g in {32,64,128,-1}
                 x {trivial, act-order}; scales log-uniform [1e-3, 5e-2]

Scales are fp16 uniform on [0.002, 0.02] except in sweep_70b.  x is fp16
N(0, 1).  Seeds: numpy PCG64 streams keyed by (workload id, K, N, g, act)
for the weights and by the same key plus M for x; single_layer uses plain
seed 0 for everything, drawn in the order qweight, qzeros, scales, x.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

WORKLOAD_IDS = {"single_layer": 0, "decode_7b": 1, "actorder_7b": 2,
                "prefill_7b": 3, "sweep_70b": 4}


def rng(*key: int) -> np.random.Generator:
    """Independent PCG64 stream for an integer key."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(0, spawn_key=tuple(int(k) for k in key))))


@dataclass
class LayerInputs:
    K: int
    N: int
    groupsize: int
    qweight: np.ndarray                 # int32 [K/8, N]
    qzeros: np.ndarray                  # int32 [G, N/8]
    scales: np.ndarray                  # float16 [G, N]
    g_idx: Optional[np.ndarray]         # int32 [K] or None (trivial)
    bias: Optional[np.ndarray]          # float16 [N] or None
    act_order: bool = False
    meta: dict = field(default_factory=dict)

    @property
    def G(self) -> int:
        return 1 if self.groupsize == -1 else self.K // self.groupsize

    @property
    def weight_bytes(self) -> int:
        """Bytes of qweight + qzeros + scales as stored in the checkpoint."""
        return self.qweight.nbytes + self.qzeros.nbytes + self.scales.nbytes


def random_words(g: np.random.Generator, shape) -> np.ndarray:
    """Uniform random 32-bit words (every nibble uniform on 0..15)."""
    return g.integers(0, 2**32, size=shape, dtype=np.uint64).astype(np.uint32).view(np.int32)


def make_layer(K: int, N: int, groupsize: int, *, act_order: bool = False,
               bias: bool = False, scale_dist: str = "uniform",
               g: Optional[np.random.Generator] = None, key=None,
               explicit_trivial_gidx: bool = False) -> LayerInputs:
    """Random GPTQ-v1 layer tensors.

    act_order: g_idx[k] = perm[k] // geff for a seeded permutation of 0..K-1.
    scale_dist: "uniform" -> U[0.002, 0.02]; "loguniform" -> logU[1e-3, 5e-2].
    """
    if g is None:
        g = rng(*(key if key is not None else (99, K, N, groupsize, int(act_order))))
    geff = K if groupsize == -1 else groupsize
    G = K // geff
    qweight = random_words(g, (K // 8, N))
    qzeros = random_words(g, (G, N // 8))
    if scale_dist == "uniform":
        s = g.uniform(0.002, 0.02, size=(G, N))
    elif scale_dist == "loguniform":
        s = np.exp(g.uniform(np.log(1e-3), np.log(5e-2), size=(G, N)))
    else:
        raise ValueError(scale_dist)
    scales = s.astype(np.float16)
    g_idx = None
    if act_order:
        perm = g.permutation(K)
        g_idx = (perm // geff).astype(np.int32)
    elif explicit_trivial_gidx:
        g_idx = (np.arange(K) // geff).astype(np.int32)
    b = g.normal(0.0, 0.1, size=N).astype(np.float16) if bias else None
    return LayerInputs(K, N, groupsize, qweight, qzeros, scales, g_idx, b, act_order)


def make_layer8(K: int, N: int, groupsize: int, *, act_order: bool = False, bias: bool = False,
                key=None) -> LayerInputs:
    """Random 8-bit GPTQ layer: qweight [K/4, N] and qzeros [G, N/4] hold
    uniform random bytes (codes and stored zeros 0..255), scales U[0.0002,
    0.002] fp16 (an 8-bit code range is 16x a 4-bit one), act-order as in
    make_layer."""
    g = rng(*(key if key is not None else (97, K, N, groupsize, int(act_order))))
    geff = K if groupsize == -1 else groupsize
    G = K // geff
    qweight = random_words(g, (K // 4, N))
    qzeros = random_words(g, (G, N // 4))
    scales = g.uniform(0.0002, 0.002, size=(G, N)).astype(np.float16)
    g_idx = (g.permutation(K) // geff).astype(np.int32) if act_order else None
    b = g.normal(0.0, 0.1, size=N).astype(np.float16) if bias else None
    return LayerInputs(K, N, groupsize, qweight, qzeros, scales, g_idx, b, act_order, {"bits": 8})


def uneven_group_index(K: int, G: int, key, empty_group: Optional[int] = None) -> np.ndarray:
    """A g_idx whose G groups hold unequal numbers of rows, scattered over K.

    Group sizes: K rows dealt to the groups with seeded random weights in
    [0.3, 1.7] (and none to `empty_group`, if given); the rows of each group
    are a seeded random subset of 0..K-1.
    """
    g = rng(*key)
    w = g.uniform(0.3, 1.7, size=G)
    if empty_group is not None:
        w[empty_group] = 0.0
    counts = np.floor(K * w / w.sum()).astype(np.int64)
    for i in np.argsort(-w)[: K - int(counts.sum())]:
        counts[i] += 1
    groups = np.repeat(np.arange(G, dtype=np.int32), counts)
    return groups[g.permutation(K)].astype(np.int32)


def activations(M: int, K: int, g: Optional[np.random.Generator] = None, key=None) -> np.ndarray:
    """x ~ N(0, 1) rounded to fp16, shape [M, K]."""
    if g is None:
        g = rng(*(key if key is not None else (98, M, K)))
    return g.standard_normal((M, K)).astype(np.float16)


def activations_bf16(M: int, K: int, key, row_scales=None) -> np.ndarray:
    """x ~ N(0, 1) (times row_scales[m] per row, if given) rounded to bf16,
    nearest-even, returned as uint16 bit patterns [M, K]."""
    g = rng(*key)
    v = g.standard_normal((M, K)).astype(np.float32)
    if row_scales is not None:
        v = (v * np.asarray(row_scales, np.float32)[:, None]).astype(np.float32)
    u = v.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16          # round to nearest, ties to even
    return u.astype(np.uint16)


def activations_f32(M: int, K: int, key, row_scales=None) -> np.ndarray:
    """x ~ N(0, 1) (times row_scales[m] per row, if given) as fp32, returned
    as uint32 bit patterns [M, K]."""
    g = rng(*key)
    v = g.standard_normal((M, K))
    if row_scales is not None:
        v = v * np.asarray(row_scales, np.float64)[:, None]
    return v.astype(np.float32).view(np.uint32)


# ------------------------------------------------------------ workloads

def single_layer():
    """M=1, K=N=1024, g=128, trivial g_idx, no bias, plain seed 0."""
    g = np.random.default_rng(0)
    layer = make_layer(1024, 1024, 128, g=g)
    x = activations(1, 1024, g=g)
    return layer, x


def workload_layer(name: str, K: int, N: int, groupsize: int, act_order: bool) -> LayerInputs:
    wid = WORKLOAD_IDS[name]
    key = (wid, K, N, groupsize & 0xFFFFFFFF, int(act_order))
    return make_layer(K, N, groupsize, act_order=act_order,
                      bias=(name == "decode_7b"),
                      scale_dist="loguniform" if name == "sweep_70b" else "uniform",
                      key=key)


def workload_x(name: str, K: int, N: int, groupsize: int, act_order: bool, M: int) -> np.ndarray:
    wid = WORKLOAD_IDS[name]
    return activations(M, K, key=(wid, K, N, groupsize & 0xFFFFFFFF, int(act_order), M))


DECODE_7B_SHAPES = [(4096, 4096), (4096, 11008), (11008, 4096), (4096, 12288)]
DECODE_7B_M = [1, 2, 4, 8]
ACTORDER_7B_SHAPES = [(4096, 11008), (11008, 4096)]
ACTORDER_7B_M = [1, 4, 16]
PREFILL_7B_SHAPES = [(4096, 4096), (4096, 11008), (11008, 4096)]
PREFILL_7B_M = [512, 2048]
SWEEP_70B_SHAPES = [(8192, 28672), (28672, 8192), (8192, 10240)]
SWEEP_70B_M = [1, 2, 4, 8, 16, 32, 64, 128, 256, 2048]
SWEEP_70B_G = [32, 64, 128, -1]


def cases(name: str):
    """(K, N, groupsize, act_order, M) tuples of a workload."""
    if name == "single_layer":
        return [(1024, 1024, 128, False, 1)]
    if name == "decode_7b":
        return [(K, N, 128, False, M) for (K, N) in DECODE_7B_SHAPES for M in DECODE_7B_M]
    if name == "actorder_7b":
        return [(K, N, 128, True, M) for (K, N) in ACTORDER_7B_SHAPES for M in ACTORDER_7B_M]
    if name == "prefill_7b":
        return [(K, N, 128, a, M) for (K, N) in PREFILL_7B_SHAPES for a in (False, True) for M in PREFILL_7B_M]
    if name == "sweep_70b":
        return [(K, N, g, a, M) for (K, N) in SWEEP_70B_SHAPES for g in SWEEP_70B_G
                for a in (False, True) for M in SWEEP_70B_M]
    raise KeyError(name)
