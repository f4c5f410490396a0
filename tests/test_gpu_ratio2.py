"""Encoder-side use of the indexer and the attention over a ratio-2 cache ([COST] §3.2: the
encoder's Full layers score the T/2 entries of their m = 2 caches; [ARCH] §3.2: the encoder
layers 2..19 write m = 2 entries). hsa_index_full, hsa_index_reindex and hsa_sparse_attn_decode
run on a cache descriptor with ratio 2 whose entries the oracle's m = 2 writer produced from 2 T
tokens of bf16 wkv / wgate; every result is checked against the oracle on the same entries.
Downstream checks are conditional, as in the other parity tests: Reindex with the kernel's pool,
attention with the kernel's indices."""
import numpy as np
import pytest

import oracle as O
from hierarchical_sparse_attention_index_gb300 import synth
from tests import parity as P

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hsa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from hierarchical_sparse_attention_index_gb300 import build
    build.build()
    import hierarchical_sparse_attention_index_gb300 as H
    H.load_library()
    return H


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def test_ratio2_full_reindex_attention(hsa):
    H = hsa
    B, nq, seed = 2, 2, 31
    n_tok = 2 * 20011                       # 20,011 entries per request
    T = n_tok // 2
    cap = (T + 7) // 8 * 8
    W = synth.w_idx_bf16(seed, 2)
    arrs = [np.zeros((B, cap, w), np.uint8) for w in (256, 32, 64, 4)]
    for b in range(B):
        out = O.cache_write_compress(P.f32(synth.latents_bf16(seed, 2, b, n_tok)),
                                     P.f32(synth.gates_bf16(seed, 2, b, n_tok)), P.f32(W), 2)
        for a, o in zip(arrs, out[:4]):
            a[b, :T] = o
    cache = H.Cache(B, cap, 2, tensors=tuple(dev(a) for a in arrs))
    oc = dict(kv_q=arrs[0], kv_s=arrs[1], ik_q=arrs[2], ik_s=arrs[3])
    q, w = synth.index_q_bf16(seed, 2, B, nq), synth.index_w(seed, 2, B, nq)
    q2, w2 = synth.index_q_bf16(seed, 8, B, nq), synth.index_w(seed, 8, B, nq)
    qa, swa = synth.attn_q_bf16(seed, 2, B, nq), synth.swa_e4m3(seed, 2, B, nq)
    vis = synth.visibility(B, nq, T)
    ws = H.new_workspace(B, nq, T)
    topk = torch.full((B, nq, 512), -7, dtype=torch.int32, device="cuda")
    pool = torch.full((B, nq, 16384), -7, dtype=torch.int32, device="cuda")
    rtop = torch.full((B, nq, 512), -7, dtype=torch.int32, device="cuda")
    out = torch.full((B, nq, 64, 512), float("nan"), device="cuda")
    H.hsa_index_full(cache, dev_bf16(q), dev(w), dev(vis), nq, T, topk, pool, ws)
    H.hsa_index_reindex(cache, dev_bf16(q2), dev(w2), dev(vis), nq, T, pool, rtop, ws)
    H.hsa_sparse_attn_decode(cache, dev_bf16(qa), rtop, dev(swa), dev(vis), nq, T, 1.0, out, ws)
    code, flags = H.hsa_get_device_status()
    assert code == 0 and flags == 0, (code, flags)
    topk, pool, rtop, out = (t.cpu().numpy() for t in (topk, pool, rtop, out))
    for b in range(B):
        K = P.dequant_index(oc, b, T)
        Km = P.dequant_main(oc, b, T)
        for i in range(nq):
            v = int(vis[b, i])
            s = O.index_scores(P.f32(q[b, i]), w[b, i], K, v)
            P.check_topk(topk[b, i], s, v, name=f"ratio2 topk b{b} q{i}")
            P.check_pool(pool[b, i], s, v, name=f"ratio2 pool b{b} q{i}")
            ref, _ = O.index_reindex(P.f32(q2[b, i]), w2[b, i], K, pool[b, i], v)
            s2 = O.index_scores(P.f32(q2[b, i]), w2[b, i], K, v)
            g = rtop[b, i]
            P.check_set_band(g[g >= 0], ref[ref >= 0], s2, f"ratio2 reindex b{b} q{i}")
            rows = O.attention_rows(Km, g, O.swa_decode(swa[b]), i, v)
            P.check_attention(out[b, i], O.sparse_attention(P.f32(qa[b, i]), rows, 1.0), f"ratio2 attn b{b} q{i}")
