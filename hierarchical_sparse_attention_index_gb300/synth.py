"""Seeded synthetic inputs for the CSA2 decode hot path.

This module produces inputs only. It holds none of the method's arithmetic: no scoring,
selection, pooling, normalisation, FP4 quantisation or attention. Both the oracle (in the
tests) and the CUDA path (tests and bench) take their inputs from here, so that the two
sides see bit-identical data.

Every array is drawn from ``numpy.random.Generator(PCG64(SeedSequence([seed, kind, layer,
request])))``. Each (tensor kind, layer, request) therefore has its own stream. A single
request of a large batch can be regenerated on its own, which the sampled full-size
parity checks rely on.

Value distributions follow the workloads the pages describe. ``N(0, v)`` names the
variance ``v``.

- Latents fed to the cache writer (``wkv``) are bf16 N(0,1). The decode caches are
  produced from them by the m=1 writer.
- ``wgate`` is bf16 N(0,2).
- The indexer projection ``W_idx`` (512x128) is bf16 N(0,1/512).
- The indexer Q (16 heads x 128) is bf16 N(0,1), with per-head weights U(0,1).
- The attention Q (64 heads x 512) is bf16 N(0,1/512).
- The SWA tail rows are N(0,1) converted to FP8 E4M3 by torch's own float8 cast. SWA KV
  production is not part of the path; these bytes are plain inputs.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

D_LATENT = 512      # main-KV latent width (head_dim)
D_INDEX = 128       # indexer head dim
H_INDEX = 16        # indexer heads
H_ATTN = 64         # attention query heads
SWA_W = 128         # sliding window

# stream kinds
_K_LATENT, _K_WIDX, _K_QIDX, _K_WIDXH, _K_QATTN, _K_SWA, _K_GATE, _K_PLANT = range(8)

_THREADS = max(1, min(16, os.cpu_count() or 1))


def _gen(seed: int, kind: int, layer: int, request: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, kind, layer, request])))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even) and return the raw uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bits to float32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_bf16(g: np.random.Generator, shape, std: float, threads: int = 1) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    if threads <= 1 or n < (1 << 22):
        x = g.standard_normal(n, dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        out[:] = f32_to_bf16_bits(x)
        return out.reshape(shape)
    # large arrays: independent child streams per chunk, filled in parallel
    chunks = threads * 4
    bounds = np.linspace(0, n, chunks + 1).astype(np.int64)
    seeds = g.bit_generator.seed_seq.spawn(chunks)

    def fill(i):
        lo, hi = bounds[i], bounds[i + 1]
        gi = np.random.Generator(np.random.PCG64(seeds[i]))
        x = gi.standard_normal(hi - lo, dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        out[lo:hi] = f32_to_bf16_bits(x)

    with ThreadPoolExecutor(threads) as ex:
        list(ex.map(fill, range(chunks)))
    return out.reshape(shape)


def latents_bf16(seed: int, layer: int, request: int, n: int, threads: int = _THREADS) -> np.ndarray:
    """[n, 512] bf16 bits, N(0,1): the wkv projection rows of one request."""
    return _normal_bf16(_gen(seed, _K_LATENT, layer, request), (n, D_LATENT), 1.0, threads)


def gates_bf16(seed: int, layer: int, request: int, n: int, threads: int = _THREADS) -> np.ndarray:
    """[n, 512] bf16 bits, N(0,2): the wgate projection rows of one request."""
    return _normal_bf16(_gen(seed, _K_GATE, layer, request), (n, D_LATENT), float(np.sqrt(2.0)), threads)


def w_idx_bf16(seed: int, layer: int) -> np.ndarray:
    """[512, 128] bf16 bits, N(0,1/512): the indexer-K projection of a KV-source layer."""
    return _normal_bf16(_gen(seed, _K_WIDX, layer, 0), (D_LATENT, D_INDEX), float(1.0 / np.sqrt(D_LATENT)))


def index_q_bf16(seed: int, layer: int, batch: int, nq: int) -> np.ndarray:
    """[B, nq, 16, 128] bf16 bits, N(0,1): the layer's indexer queries."""
    return _normal_bf16(_gen(seed, _K_QIDX, layer, 0), (batch, nq, H_INDEX, D_INDEX), 1.0)


def index_w(seed: int, layer: int, batch: int, nq: int) -> np.ndarray:
    """[B, nq, 16] float32, U(0,1): the layer's per-head indexer weights."""
    return _gen(seed, _K_WIDXH, layer, 0).random((batch, nq, H_INDEX), dtype=np.float32)


def attn_q_bf16(seed: int, layer: int, batch: int, nq: int) -> np.ndarray:
    """[B, nq, 64, 512] bf16 bits, N(0,1/512): the layer's attention queries."""
    return _normal_bf16(_gen(seed, _K_QATTN, layer, 0), (batch, nq, H_ATTN, D_LATENT),
                        float(1.0 / np.sqrt(D_LATENT)))


def swa_e4m3(seed: int, layer: int, batch: int, nq: int) -> np.ndarray:
    """[B, W+nq-1, 512] uint8: N(0,1) rows cast to FP8 E4M3 by torch's float8 conversion."""
    import torch
    x = _gen(seed, _K_SWA, layer, 0).standard_normal((batch, SWA_W + nq - 1, D_LATENT), dtype=np.float32)
    return torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def visibility(batch: int, nq: int, T: int) -> np.ndarray:
    """[B, nq] int32: query i of a request sees positions [0, T - nq + 1 + i)."""
    v = np.arange(nq, dtype=np.int32) + np.int32(T - nq + 1)
    return np.broadcast_to(v, (batch, nq)).copy()


def plant_clusters(latent_bits: np.ndarray, w_idx_bits: np.ndarray, q_bits: np.ndarray,
                   w: np.ndarray, n_clusters: int, seed: int, request: int) -> np.ndarray:
    """Plant ``n_clusters`` runs of 8 adjacent, 8-aligned positions whose latent points along
    ``W_idx @ u``, with ``u = sum_h w_h q_h`` built from the Full layer's indexer query.

    After the cache writer normalises such a latent and projects it, its indexer key is
    close to ``sqrt(512) * u / |u|``, which makes every planted position score far above
    the N(0,1) background. Returns the sorted planted positions; ``latent_bits`` is
    modified in place.
    """
    T = latent_bits.shape[0]
    g = _gen(seed, _K_PLANT, 0, request)
    nblk = T // 8
    blocks = np.sort(g.choice(nblk, size=n_clusters, replace=False))
    q = bf16_bits_to_f32(q_bits).astype(np.float64)            # [16, 128]
    u = (w.astype(np.float64)[:, None] * q).sum(axis=0)       # [128]
    W = bf16_bits_to_f32(w_idx_bits).astype(np.float64)        # [512, 128]
    direction = W @ u
    direction /= np.sqrt(np.mean(direction ** 2))
    jitter = g.standard_normal((n_clusters, 8, D_LATENT)) * 0.05
    rows = direction[None, None, :] * (1.0 + jitter)
    pos = (blocks[:, None] * 8 + np.arange(8)[None, :]).reshape(-1)
    latent_bits[pos] = f32_to_bf16_bits(rows.reshape(-1, D_LATENT).astype(np.float32))
    return pos


@dataclass
class DecodeConfig:
    """Shape of one decode workload."""
    name: str
    seed: int
    batch: int
    T: int
    nq: int
    layers: list = field(default_factory=list)   # decoder layer ids that run in one step
    planted: int = 0

    @property
    def entries(self) -> int:
        return self.T


# The five workloads of the pages (decode ones here; the m=2 cache write below).
CFG0 = DecodeConfig("b1_t32k_full_reindex", 0, 1, 32768, 1, [20, 24])
CFG1 = DecodeConfig("b32_t128k_20layers", 1000, 32, 131072, 1, list(range(20, 40)))
CFG2 = DecodeConfig("b4_t1m_planted", 2000, 4, 1 << 20, 1, [20, 24, 28, 32, 36], planted=64)
CFG4 = DecodeConfig("b64_nq5_t64k_verify", 4000, 64, 65536, 5, list(range(20, 40)))

CFG3_SEED = 3000
CFG3_LAYERS = (2, 8, 14)
CFG3_TOKENS = 65536
