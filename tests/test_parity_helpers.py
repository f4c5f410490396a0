"""CPU checks of the parity helpers that the full-size GPU tests lean on: the pooled oracle
writer must give exactly the single-call writer's bytes (entries depend only on their own
tokens), and the on-demand main-KV rows must equal the full dequantisation."""
import multiprocessing as mp

import numpy as np

import oracle as O
from hierarchical_sparse_attention_index_gb300 import synth
from tests import parity as P


def test_pooled_writer_matches_single_call():
    n = 300
    wkv = synth.latents_bf16(5, 2, 0, n)
    wg = synth.gates_bf16(5, 2, 0, n)
    W = synth.w_idx_bf16(5, 2)
    with mp.get_context("spawn").Pool(2) as pool:
        for m, g in ((1, None), (2, wg)):
            got = P.oracle_write(pool, wkv, g, W, m=m, keep=True, chunk=64)
            ref = O.cache_write_compress(P.f32(wkv), None if g is None else P.f32(g), P.f32(W), m)
            assert len(got) == 6
            for a, b in zip(got, ref):
                assert np.array_equal(a, b)


def test_main_rows_on_demand():
    n = 40
    wkv = synth.latents_bf16(6, 20, 0, n)
    W = synth.w_idx_bf16(6, 20)
    kv_q, kv_s, _, _, _, _ = O.cache_write_compress(P.f32(wkv), None, P.f32(W), 1)
    full = O.main_kv_dequant(kv_q, kv_s)
    rows = P.MainRows(kv_q, kv_s)
    sel = [3, 17, 39, 0]
    assert np.array_equal(rows[sel], full[sel])
