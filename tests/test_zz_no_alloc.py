"""The no-allocation Reindex entry point (hsa_index_reindex_noalloc), called through the C ABI.

It serves callers that cannot allocate device memory, such as plugins limited to the buffers
they are handed, or code inside an allocator-managed arena. The fused Reindex kernel keeps its
exchange in shared memory, so the call uses no scratch memory at all. The tests check that two
calls in a row give exactly the output of the workspace-based hsa_index_reindex, within the
oracle's top-k band, and that a many-row request (36 rows) matches it too. This file is
collected last and passes both on its own in a fresh process and after the other tests."""
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


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def test_reindex_noalloc_matches_workspace_reindex(hsa):
    H = hsa
    B, T, nq, seed = 3, 12344, 2, 21
    oc = P.oracle_cache(seed, 20, B, T, T)
    cache = H.Cache(B, T, 1, tensors=tuple(_dev(oc[k]) for k in ("kv_q", "kv_s", "ik_q", "ik_s")))
    vis = _dev(synth.visibility(B, nq, T))
    q20, w20 = synth.index_q_bf16(seed, 20, B, nq), synth.index_w(seed, 20, B, nq)
    q24, w24 = synth.index_q_bf16(seed, 24, B, nq), synth.index_w(seed, 24, B, nq)
    ws = H.new_workspace(B, nq, T)
    top20 = torch.empty(B, nq, 512, dtype=torch.int32, device="cuda")
    pool = torch.empty(B, nq, 16384, dtype=torch.int32, device="cuda")
    H.hsa_index_full(cache, _dev_bf16(q20), _dev(w20), vis, nq, T, top20, pool, ws)
    ref = torch.full((B, nq, 512), -7, dtype=torch.int32, device="cuda")
    H.hsa_index_reindex(cache, _dev_bf16(q24), _dev(w24), vis, nq, T, pool, ref, ws)
    pool_h, ref_h = pool.cpu().numpy(), ref.cpu().numpy()
    vis_h = synth.visibility(B, nq, T)
    for call in range(2):
        out = torch.full((B, nq, 512), -7, dtype=torch.int32, device="cuda")
        H.hsa_index_reindex_noalloc(cache, _dev_bf16(q24), _dev(w24), vis, nq, T, pool, out)
        code, flags = H.hsa_get_device_status()
        assert code == 0 and flags == 0, (call, code, flags)
        out_h = out.cpu().numpy()
        assert np.array_equal(out_h, ref_h), f"call {call}: differs from hsa_index_reindex"
        for b in range(B):
            K = P.dequant_index(oc, b, T)
            for i in range(nq):
                v = int(vis_h[b, i])
                s = O.index_scores(P.f32(q24[b, i]), w24[b, i], K, v)
                o, _ = O.index_reindex(P.f32(q24[b, i]), w24[b, i], K, pool_h[b, i], v)
                g = out_h[b, i]
                P.check_set_band(g[g >= 0], o[o >= 0], s, f"noalloc call {call} b{b} q{i}")


def test_reindex_noalloc_many_rows(hsa):
    H = hsa
    B, nq, T, seed = 9, 4, 3000, 5            # 36 rows
    oc = P.oracle_cache(seed, 20, B, T, T)
    cache = H.Cache(B, T, 1, tensors=tuple(_dev(oc[k]) for k in ("kv_q", "kv_s", "ik_q", "ik_s")))
    vis = _dev(synth.visibility(B, nq, T))
    q20, w20 = synth.index_q_bf16(seed, 20, B, nq), synth.index_w(seed, 20, B, nq)
    q24, w24 = synth.index_q_bf16(seed, 24, B, nq), synth.index_w(seed, 24, B, nq)
    ws = H.new_workspace(B, nq, T)
    top20 = torch.empty(B, nq, 512, dtype=torch.int32, device="cuda")
    pool = torch.empty(B, nq, 16384, dtype=torch.int32, device="cuda")
    H.hsa_index_full(cache, _dev_bf16(q20), _dev(w20), vis, nq, T, top20, pool, ws)
    ref = torch.full((B, nq, 512), -7, dtype=torch.int32, device="cuda")
    H.hsa_index_reindex(cache, _dev_bf16(q24), _dev(w24), vis, nq, T, pool, ref, ws)
    out = torch.full((B, nq, 512), -7, dtype=torch.int32, device="cuda")
    H.hsa_index_reindex_noalloc(cache, _dev_bf16(q24), _dev(w24), vis, nq, T, pool, out)
    code, flags = H.hsa_get_device_status()
    assert code == 0 and flags == 0, (code, flags)
    assert torch.equal(out, ref)
