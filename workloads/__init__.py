"""Seeded synthetic inputs shaped like the pages' decode workloads.

This module is shared by the oracle side and the CUDA side.  It only draws
random numbers and lays them out; it holds none of the method's arithmetic
(no cosine, threshold, softmax or attention).  Everything is seeded, so a
(config, seed, device) triple always gives the same tensors.  The CPU and CUDA
torch generators give different streams, so parity tests always hand both
sides the very same tensors (generated once, then copied).

Shapes follow the models the CLO page evaluates ("CLO: CPU-Light KVCache
Offloading", section 2: Llama3-8B with 32 layers, 32 query / 8 KV heads and
Qwen2.5-14B with 48 layers, 40 query / 8 KV heads; sparsity 10%, eta = 0.8,
n = 3) and the Llama-2-7B many-request paged decode of the NEO page ("Neo:
Saving GPU Memory Crisis with CPU Offloading for Online LLM Inference",
experimental setup).  Real traces (RULER, LongBench, Azure code, OpenAI
summarisation) are not available; these distributions stand in for them.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional

import numpy as np
import torch

ETA = 0.8
N_EXP = 3.0
SPARSITY_DIV = 10  # top-k = floor(T / 10): 10% sparsity
HEAD_DIM = 128
BLOCK_SIZE = 16


@dataclass(frozen=True)
class HybridConfig:
    """One CLO decode workload (hybrid Cache Buffer + Persistent Cache)."""
    name: str
    B: int
    L: int
    Hq: int
    Hkv: int
    T: int
    Np: int
    d: int = HEAD_DIM
    qmode: str = "mix"           # "mix": q = 0.8*label + 0.6*N(0,1)
                                 # "cos": cos(q, label) ~ U(c_lo, c_hi) per head
    c_lo: float = 0.7
    c_hi: float = 0.9
    low_frac: float = 0.0        # fraction of heads drawn from [c_lo-0.2, c_hi-0.2]
    smode: str = "uniform"       # importance s ~ U(0,1) ("uniform"), Beta(0.5, 2) ("beta"),
                                 # or s = 1 on every head ("one": tau = eta)
    label_reset: bool = False    # the benchmark restores the drawn labels every step, so the
                                 # same groups miss again (a miss copies q into the label)
    miss_fill: str = ""          # "host" / "device": the benchmark fills the missed heads'
                                 # rows from a full KV copy there after each lookup
    addressing: str = "token"    # "token": C = T slots, idx = positions in [0, T)
                                 # "compact": C = k slots, idx = permutation of [0, k)
    ring: int = 0                # >0: only `ring` physical layer buffers, reused cyclically
    idx_order: str = "random"    # "random": idx in random order; "sorted": ascending, as
                                 # the top-k retrieval writes it
    seed: int = 1234

    @property
    def k(self) -> int:
        return self.T // SPARSITY_DIV

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def C(self) -> int:
        return self.T if self.addressing == "token" else self.k


@dataclass(frozen=True)
class PagedConfig:
    """Dense paged decode attention over many requests."""
    name: str
    B: int
    Hq: int
    Hkv: int
    ctx_lo: int
    ctx_hi: int
    d: int = HEAD_DIM
    block_size: int = BLOCK_SIZE
    seed: int = 1238

    @property
    def max_blocks(self) -> int:
        return -(-self.ctx_hi // self.block_size)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv


CONFIGS = {
    # Tiny CLO step: batch 1, one layer, GQA 4, context 1024, k = 102, 2 persistent heads.
    "tiny": HybridConfig("tiny", B=1, L=1, Hq=32, Hkv=8, T=1024, Np=2,
                         qmode="mix", smode="uniform", seed=1234),
    # Llama3-8B-shaped single layer: batch 8, context 32K.
    "llama3_8b_layer_b8_32k": HybridConfig(
        "llama3_8b_layer_b8_32k", B=8, L=1, Hq=32, Hkv=8, T=32768, Np=2,
        qmode="cos", c_lo=0.7, c_hi=0.9, smode="beta", seed=1235),
    # Llama3-8B-shaped full decode step, context 128K, batch 1 and batch 4.
    "llama3_8b_step_b1_128k": HybridConfig(
        "llama3_8b_step_b1_128k", B=1, L=32, Hq=32, Hkv=8, T=131072, Np=2,
        qmode="mix", smode="uniform", seed=1236),
    "llama3_8b_step_b4_128k": HybridConfig(
        "llama3_8b_step_b4_128k", B=4, L=32, Hq=32, Hkv=8, T=131072, Np=2,
        qmode="mix", smode="uniform", seed=1236),
    # The batch-8 layer with each head's Cache Buffer indices in ascending
    # order (as the top-k retrieval writes them): measured beside the default.
    "llama3_8b_layer_b8_32k_sorted": HybridConfig(
        "llama3_8b_layer_b8_32k_sorted", B=8, L=1, Hq=32, Hkv=8, T=32768, Np=2,
        qmode="cos", c_lo=0.7, c_hi=0.9, smode="beta", idx_order="sorted", seed=1235),
    # The batch-8 layer with misses at the page's head-level hit rate (CLO
    # section 5, Table 4: 79% on average).  With the configured importance
    # draws every KV head's tau sits near -1 and nothing misses, so here every
    # query head has s = 1 (tau = eta = 0.8, the top of the threshold chain)
    # and the query/label cosines are drawn from U(0.725, 0.925): the mean
    # over a GQA-4 group falls below 0.8 for about 20% of the groups.
    "llama3_8b_layer_b8_32k_miss": HybridConfig(
        "llama3_8b_layer_b8_32k_miss", B=8, L=1, Hq=32, Hkv=8, T=32768, Np=2,
        qmode="cos", c_lo=0.725, c_hi=0.925, smode="one", label_reset=True, seed=1239),
    # The same with the miss path after each lookup: the missed heads' top-k
    # rows fetched from the full KV copy in pinned host memory into the Cache
    # Buffer rows the next attention reads (CLO section 3, Fig. 7).
    "llama3_8b_layer_b8_32k_miss_fill": HybridConfig(
        "llama3_8b_layer_b8_32k_miss_fill", B=8, L=1, Hq=32, Hkv=8, T=32768, Np=2,
        qmode="cos", c_lo=0.725, c_hi=0.925, smode="one", label_reset=True,
        miss_fill="host", seed=1239),
    # The batch-1, 128K-context step (the page's single-layer setting: Llama3-8B,
    # BSZ 1, 128K, top-k 10%) with misses at the page's hit rate and the missed
    # heads' rows fetched from a full KV copy in pinned host memory.  Every
    # layer has its own buffers (17 GB of pinned host memory for the full
    # copies): the same heads miss every step, and with fewer physical layers
    # their rows would be read from L2, not over the host link.
    "llama3_8b_step_b1_128k_miss_fill": HybridConfig(
        "llama3_8b_step_b1_128k_miss_fill", B=1, L=32, Hq=32, Hkv=8, T=131072, Np=2,
        qmode="cos", c_lo=0.725, c_hi=0.925, smode="one", label_reset=True,
        miss_fill="host", seed=1240),
    # Qwen2.5-14B-shaped decode step: 48 layers, GQA 5, batch 16, context 64K,
    # 15% of heads with cosine ~0.6; a ring of 8 physical layer buffers.
    "qwen25_14b_step_b16_64k": HybridConfig(
        "qwen25_14b_step_b16_64k", B=16, L=48, Hq=40, Hkv=8, T=65536, Np=1,
        qmode="cos", c_lo=0.7, c_hi=0.9, low_frac=0.15, smode="beta", ring=8,
        seed=1237),
}

PAGED_CONFIGS = {
    # Llama-2-7B shape, 32 MHA heads, batch 256, context U[128, 4096], 16-token blocks.
    "paged_llama2_7b_b256": PagedConfig("paged_llama2_7b_b256", B=256, Hq=32,
                                        Hkv=32, ctx_lo=128, ctx_hi=4096, seed=1238),
}


# Miss-path fill: the Cache Buffer rows of every non-persistent KV head of the
# Llama3-8B-shaped batch-8 layer refilled from the full KV copy, which sits in
# pinned host memory (read over the host link) or in HBM.
FILL_CONFIGS = {
    "fill_c2c_llama3_8b_b8_32k": ("llama3_8b_layer_b8_32k", "host"),
    "fill_hbm_llama3_8b_b8_32k": ("llama3_8b_layer_b8_32k", "device"),
}


# Top-k retrieval: every KV head of the Llama3-8B-shaped batch-8 layer ranks
# all of its 32768 keys against its query group and keeps the top 10%.
TOPK_CONFIGS = {
    "topk_llama3_8b_b8_32k": "llama3_8b_layer_b8_32k",
}


def small_hybrid(name="small", **kw) -> HybridConfig:
    """A reduced workload for quick parity runs (any field overridable)."""
    base = dict(B=2, L=1, Hq=32, Hkv=8, T=1000, Np=2, qmode="mix",
                smode="uniform", seed=4321)
    base.update(kw)
    return HybridConfig(name, **base)


def small_paged(name="small_paged", **kw) -> PagedConfig:
    base = dict(B=6, Hq=8, Hkv=8, ctx_lo=1, ctx_hi=300, seed=8765)
    base.update(kw)
    return PagedConfig(name, **base)


def _seed(*parts: int) -> int:
    """Derives a 63-bit seed from integer parts (splitmix64-style mixing)."""
    x = 0x9E3779B97F4A7C15
    for p in parts:
        x = (x ^ (int(p) & 0xFFFFFFFFFFFFFFFF)) & 0xFFFFFFFFFFFFFFFF
        x = (x * 0xBF58476D1CE4E5B9) & 0xFFFFFFFFFFFFFFFF
        x ^= x >> 31
    return x & 0x7FFFFFFFFFFFFFFF


def _torch_gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(seed)
    return g


def _np_rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


# --- per-layer small arrays (numpy, identical on every device) -------------

def importance(cfg: HybridConfig, layer: int) -> np.ndarray:
    """Importance scores s of the query heads of one layer, float32 [Hq]."""
    rng = _np_rng(_seed(cfg.seed, layer, 1))
    if cfg.smode == "uniform":
        s = rng.uniform(0.0, 1.0, size=cfg.Hq)
    elif cfg.smode == "beta":
        s = rng.beta(0.5, 2.0, size=cfg.Hq)
    elif cfg.smode == "one":
        s = np.ones(cfg.Hq)
    else:
        raise ValueError(cfg.smode)
    return s.astype(np.float32)


def persist_ids(cfg: HybridConfig, layer: int) -> np.ndarray:
    """The layer's persistent KV heads, int32 [Np], distinct, in random order."""
    rng = _np_rng(_seed(cfg.seed, layer, 2))
    return rng.permutation(cfg.Hkv)[: cfg.Np].astype(np.int32)


def persist_mask(cfg: HybridConfig, layer: int) -> np.ndarray:
    """uint8 [Hkv]: 1 where the KV head is persistent."""
    m = np.zeros(cfg.Hkv, dtype=np.uint8)
    m[persist_ids(cfg, layer)] = 1
    return m


# --- bulk tensors (torch, on the requested device) -------------------------

def queries_and_labels(cfg: HybridConfig, layer: int, device="cpu"):
    """(q, labels), fp16 [B][Hq][d].  labels ~ N(0,1).

    qmode "mix": q = 0.8*label + 0.6*N(0,1).
    qmode "cos": q = c*label + sqrt(1-c^2)*n_perp, n_perp orthogonal to the
    label with the label's norm, c ~ U(c_lo, c_hi) per (b, head) (a fraction
    low_frac of heads drawn 0.2 lower).
    """
    g = _torch_gen(device, _seed(cfg.seed, layer, 3))
    shape = (cfg.B, cfg.Hq, cfg.d)
    lab = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    noise = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if cfg.qmode == "mix":
        q = 0.8 * lab + 0.6 * noise
    elif cfg.qmode == "cos":
        u = torch.rand((cfg.B, cfg.Hq, 1), generator=g, device=device)
        low = torch.rand((cfg.B, cfg.Hq, 1), generator=g, device=device) < cfg.low_frac
        c = cfg.c_lo + (cfg.c_hi - cfg.c_lo) * u - 0.2 * low.float()
        lhat = lab / lab.norm(dim=-1, keepdim=True)
        perp = noise - (noise * lhat).sum(-1, keepdim=True) * lhat
        perp = perp * (lab.norm(dim=-1, keepdim=True) / perp.norm(dim=-1, keepdim=True))
        q = c * lab + torch.sqrt(1.0 - c * c) * perp
    else:
        raise ValueError(cfg.qmode)
    return q.to(torch.float16), lab.to(torch.float16)


def cache_buffer(cfg: HybridConfig, layer: int, device="cpu"):
    """(cbK, cbV, idx): Cache Buffer fp16 [B][Hkv][C][d] ~ N(0,1) and the
    per-(b, KV head) row indices int32 [B][Hkv][k], distinct, unsorted."""
    g = _torch_gen(device, _seed(cfg.seed, layer, 4))
    shape = (cfg.B, cfg.Hkv, cfg.C, cfg.d)
    cbK = torch.randn(shape, generator=g, device=device, dtype=torch.float16)
    cbV = torch.randn(shape, generator=g, device=device, dtype=torch.float16)
    keys = torch.rand((cfg.B * cfg.Hkv, cfg.C), generator=g, device=device)
    idx = keys.argsort(dim=1)[:, : cfg.k].to(torch.int32)
    if cfg.idx_order == "sorted":
        idx = idx.sort(dim=1).values
    return cbK, cbV, idx.reshape(cfg.B, cfg.Hkv, cfg.k).contiguous()


def persistent_cache(cfg: HybridConfig, layer: int, device="cpu"):
    """(pK, pV): Persistent Cache fp16 [B][Np][T][d] ~ N(0,1)."""
    g = _torch_gen(device, _seed(cfg.seed, layer, 5))
    shape = (cfg.B, cfg.Np, cfg.T, cfg.d)
    pK = torch.randn(shape, generator=g, device=device, dtype=torch.float16)
    pV = torch.randn(shape, generator=g, device=device, dtype=torch.float16)
    return pK, pV


def full_kv(cfg: HybridConfig, layer: int, device="cpu"):
    """(srcK, srcV): the full KV copy of every head, fp16 [B][Hkv][T][d] ~ N(0,1)
    (what the miss-path fill reads from)."""
    g = _torch_gen(device, _seed(cfg.seed, layer, 6))
    shape = (cfg.B, cfg.Hkv, cfg.T, cfg.d)
    srcK = torch.randn(shape, generator=g, device=device, dtype=torch.float16)
    srcV = torch.randn(shape, generator=g, device=device, dtype=torch.float16)
    return srcK, srcV


def fill_selection(cfg: HybridConfig, layer: int, device="cpu"):
    """(tok, slot) int32 [B][Hkv][k]: each head's new top-k token set (k
    distinct tokens of [0, T), unsorted) and the Cache Buffer row of each (the
    token itself with token addressing, a permutation of [0, k) with compact
    addressing)."""
    g = _torch_gen(device, _seed(cfg.seed, layer, 7))
    keys = torch.rand((cfg.B * cfg.Hkv, cfg.T), generator=g, device=device)
    tok = keys.argsort(dim=1)[:, : cfg.k].to(torch.int32).reshape(cfg.B, cfg.Hkv, cfg.k)
    if cfg.addressing == "token":
        slot = tok.clone()
    else:
        keys = torch.rand((cfg.B * cfg.Hkv, cfg.k), generator=g, device=device)
        slot = keys.argsort(dim=1).to(torch.int32).reshape(cfg.B, cfg.Hkv, cfg.k)
    return tok.contiguous(), slot.contiguous()


def paged_context_lengths(cfg: PagedConfig) -> np.ndarray:
    """int32 [B], uniform integers in [ctx_lo, ctx_hi]."""
    rng = _np_rng(_seed(cfg.seed, 1))
    return rng.integers(cfg.ctx_lo, cfg.ctx_hi + 1, size=cfg.B).astype(np.int32)


def paged_block_table(cfg: PagedConfig) -> np.ndarray:
    """int32 [B][max_blocks]: a random permutation of all B*max_blocks pool
    blocks (the pool is sized for the longest possible context)."""
    rng = _np_rng(_seed(cfg.seed, 2))
    nb = cfg.B * cfg.max_blocks
    return rng.permutation(nb).astype(np.int32).reshape(cfg.B, cfg.max_blocks)


def paged_inputs(cfg: PagedConfig, device="cpu"):
    """(q, kc, vc, block_table, ctx_len): q fp16 [B][Hq][d]; kc/vc fp16
    [num_blocks][Hkv][block_size][d] ~ N(0,1); block table and lengths int32."""
    g = _torch_gen(device, _seed(cfg.seed, 3))
    nb = cfg.B * cfg.max_blocks
    q = torch.randn((cfg.B, cfg.Hq, cfg.d), generator=g, device=device, dtype=torch.float16)
    shape = (nb, cfg.Hkv, cfg.block_size, cfg.d)
    kc = torch.randn(shape, generator=g, device=device, dtype=torch.float16)
    vc = torch.randn(shape, generator=g, device=device, dtype=torch.float16)
    bt = torch.from_numpy(paged_block_table(cfg)).to(device)
    ctx = torch.from_numpy(paged_context_lengths(cfg)).to(device)
    return q, kc, vc, bt, ctx
