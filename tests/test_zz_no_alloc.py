"""The allocation-free Full indexer (hsa_index_full_noalloc), called through the C ABI.

It serves callers that cannot allocate device memory, such as plugins limited to the buffers
they are handed, code inside an arena an inference server planned in advance, or loops that
must never wait on an allocator. Its scratch is a fixed array inside the library that every
call shares. The tests check that two calls in a row give exactly the output of the
workspace-based hsa_index_full (the same kernels), that both lie within the oracle's top-k band,
and that sizes beyond the fixed array are refused before anything is launched. This file is
collected last; it passes on its own in a fresh process and after the other tests."""
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


def test_full_noalloc_matches_workspace_full(hsa):
    H = hsa
    B, T, nq, seed = 3, 12344, 2, 21
    oc = P.oracle_cache(seed, 20, B, T, T)
    cache = H.Cache(B, T, 1, tensors=tuple(_dev(oc[k]) for k in ("kv_q", "kv_s", "ik_q", "ik_s")))
    vis_h = synth.visibility(B, nq, T)
    vis = _dev(vis_h)
    q20, w20 = synth.index_q_bf16(seed, 20, B, nq), synth.index_w(seed, 20, B, nq)
    ws = H.new_workspace(B, nq, T)
    ref_top = torch.full((B, nq, 512), -7, dtype=torch.int32, device="cuda")
    ref_pool = torch.full((B, nq, 16384), -7, dtype=torch.int32, device="cuda")
    H.hsa_index_full(cache, _dev_bf16(q20), _dev(w20), vis, nq, T, ref_top, ref_pool, ws)
    for call in range(2):
        top = torch.full((B, nq, 512), -7, dtype=torch.int32, device="cuda")
        pool = torch.full((B, nq, 16384), -7, dtype=torch.int32, device="cuda")
        H.hsa_index_full_noalloc(cache, _dev_bf16(q20), _dev(w20), vis, nq, T, top, pool)
        code, flags = H.hsa_get_device_status()
        assert code == 0 and flags == 0, (call, code, flags)
        assert torch.equal(top, ref_top), f"call {call}: top-512 differs from hsa_index_full"
        assert torch.equal(pool, ref_pool), f"call {call}: pool differs from hsa_index_full"
        top_h, pool_h = top.cpu().numpy(), pool.cpu().numpy()
        for b in range(B):
            K = P.dequant_index(oc, b, T)
            for i in range(nq):
                v = int(vis_h[b, i])
                s = O.index_scores(P.f32(q20[b, i]), w20[b, i], K, v)
                P.check_topk(top_h[b, i], s, v, name=f"noalloc call {call} b{b} q{i}")
                P.check_pool(pool_h[b, i], s, v, name=f"noalloc pool call {call} b{b} q{i}")


def test_full_noalloc_refuses_sizes_beyond_the_array(hsa):
    H = hsa
    # batch 64 x 1,048,576 positions needs far more scratch than the fixed array holds; the call
    # is refused on the host, so the (never dereferenced) cache buffers can stay tiny
    z = torch.zeros(64, dtype=torch.uint8, device="cuda")
    cache = H.Cache.__new__(H.Cache)
    cache.desc = H.hsa_cache(64, 1, 1 << 20, 0, 0, z.data_ptr(), z.data_ptr(), z.data_ptr(), z.data_ptr())
    buf = torch.zeros(64, dtype=torch.int32, device="cuda")
    with pytest.raises(H.HsaError) as e:
        H.hsa_index_full_noalloc(cache, buf, buf, buf, 1, 1 << 20, buf, buf)
    assert e.value.code == 4   # HSA_ERR_WORKSPACE
