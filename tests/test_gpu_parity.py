"""GPU parity: every entry point of include/hsa.h, called through the C ABI, against the fp64
oracle on the same seeded inputs. Sizes span several tiles and a ragged tail, and the edge
cases (tiny and non-multiple contexts, contexts shorter than the window, multi-query verify
blocks, out-of-range indices) are covered. Downstream checks are conditional: reindex is
checked with the kernel's own pool and attention with the kernel's own indices, so a legal
near-tie upstream cannot cascade."""
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


def gpu_cache(H, oc, cap, fmt=O.SCALE_E8M0):
    B = oc["kv_q"].shape[0]
    return H.Cache(B, cap, 1, fmt, tensors=(dev(oc["kv_q"]), dev(oc["kv_s"]), dev(oc["ik_q"]), dev(oc["ik_s"])))


def round8(n):
    return max(8, (n + 7) // 8 * 8)


# ------------------------------------------------------------------ cache write
@pytest.mark.parametrize("fmt", [O.SCALE_E8M0, O.SCALE_E4M3])
def test_cache_write_m1(hsa, fmt):
    H = hsa
    seed, B, n, cap = 11, 2, 777, 1024
    starts = np.array([0, 100], np.int64)
    wkv = np.stack([synth.latents_bf16(seed, 20, b, n) for b in range(B)])
    W = synth.w_idx_bf16(seed, 20)
    cache = H.Cache(B, cap, 1, fmt)
    H.hsa_cache_write_compress(cache, dev_bf16(wkv), None, dev_bf16(W), n, dev(starts))
    code, flags = H.hsa_get_device_status()
    assert code == 0 and flags == 0
    g = [t.cpu().numpy() for t in (cache.kv_q, cache.kv_s, cache.ik_q, cache.ik_s)]
    for b in range(B):
        kv_q, kv_s, ik_q, ik_s, lat, K = O.cache_write_compress(P.f32(wkv[b]), None, P.f32(W), 1, fmt)
        ent = np.arange(starts[b], starts[b] + n)
        P.check_write((lat, K, P.f32(W).astype(np.float64)), (kv_q, kv_s, ik_q, ik_s),
                     [x[b] for x in g], ent, fmt, f"m1 b{b}")
        untouched = np.setdiff1d(np.arange(cap), ent)
        assert not g[0][b][untouched].any() and not g[2][b][untouched].any()


@pytest.mark.parametrize("fmt", [O.SCALE_E8M0, O.SCALE_E4M3])
def test_cache_write_m2(hsa, fmt):
    H = hsa
    seed, n = 12, 4097                       # odd: the trailing token is not written
    wkv = synth.latents_bf16(seed, 2, 0, n)[None]
    wg = synth.gates_bf16(seed, 2, 0, n)[None]
    W = synth.w_idx_bf16(seed, 2)
    cache = H.Cache(1, 2056, 2, fmt)
    H.hsa_cache_write_compress(cache, dev_bf16(wkv), dev_bf16(wg), dev_bf16(W), n, None)
    g = [t.cpu().numpy()[0] for t in (cache.kv_q, cache.kv_s, cache.ik_q, cache.ik_s)]
    kv_q, kv_s, ik_q, ik_s, lat, K = O.cache_write_compress(P.f32(wkv[0]), P.f32(wg[0]), P.f32(W), 2, fmt)
    assert lat.shape[0] == 2048
    P.check_write((lat, K, P.f32(W).astype(np.float64)), (kv_q, kv_s, ik_q, ik_s), g, np.arange(2048), fmt, "m2")
    assert not g[0][2048:].any()


@pytest.mark.parametrize("m", [1, 2])
def test_cache_write_rope(hsa, m):
    """HSA_CACHE_ROPE: main KV holds the latent with its last 64 dims turned by the entry's
    position (positions up to about 2^20, where a float32 angle would be off by ~0.06 rad);
    indexer K is the no-RoPE projection. Both against the oracle's writer with rope_pos."""
    H = hsa
    seed, n, B = 13, 1600, 2
    ne = n // m
    cap = 1 << 20
    starts = np.array([0, cap - ne - 8], np.int64)
    wkv = np.stack([synth.latents_bf16(seed, 20, b, n) for b in range(B)])
    wg = np.stack([synth.gates_bf16(seed, 20, b, n) for b in range(B)]) if m == 2 else None
    W = synth.w_idx_bf16(seed, 20)
    cache = H.Cache(B, cap, m, flags=H.HSA_CACHE_ROPE)
    H.hsa_cache_write_compress(cache, dev_bf16(wkv), dev_bf16(wg) if m == 2 else None, dev_bf16(W), n, dev(starts))
    code, flags = H.hsa_get_device_status()
    assert code == 0 and flags == 0
    for b in range(B):
        ent = np.arange(starts[b], starts[b] + ne)
        kv_q, kv_s, ik_q, ik_s, lat, K = O.cache_write_compress(P.f32(wkv[b]), None if m == 1 else P.f32(wg[b]),
                                                                P.f32(W), m, rope_pos=ent)
        g = [t[b, starts[b]:starts[b] + ne].cpu().numpy() for t in (cache.kv_q, cache.kv_s, cache.ik_q, cache.ik_s)]
        P.check_write((lat, K, P.f32(W).astype(np.float64)), (kv_q, kv_s, ik_q, ik_s), g, np.arange(ne),
                      O.SCALE_E8M0, f"rope m{m} b{b}")


def test_cache_write_rejects_bad_args(hsa):
    H = hsa
    cache = H.Cache(1, 64, 2)
    x = torch.zeros(1, 16, 512, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(512, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(H.HsaError):          # ratio 2 needs wgate
        H.hsa_cache_write_compress(cache, x, None, W, 16)
    starts = torch.tensor([60], dtype=torch.int64, device="cuda")
    H.hsa_cache_write_compress(cache, x, x, W, 16, starts)   # entries 60..67: 64..67 are past capacity
    code, flags = H.hsa_get_device_status()
    assert flags & H.HSA_FLAG_WRITE_RANGE


# ------------------------------------------------------------------ Full indexer
FULL_CASES = [  # (B, T, nq)
    (1, 32768, 1), (3, 5000, 1), (1, 1, 1), (1, 7, 1), (1, 9, 1), (1, 511, 1), (1, 513, 1),
    (1, 16385, 1), (2, 4100, 5), (1, 20000, 2), (1, 3000, 8),
]


def _full_case(H, B, T, nq, seed=0):
    cap = round8(T)
    oc = P.oracle_cache(seed, 20, B, T, cap)
    q = synth.index_q_bf16(seed, 20, B, nq)
    w = synth.index_w(seed, 20, B, nq)
    vis = synth.visibility(B, nq, T)
    cache = gpu_cache(H, oc, cap)
    ws = H.new_workspace(B, nq, T)
    topk = torch.full((B, nq, 512), -7, dtype=torch.int32, device="cuda")
    pool = torch.full((B, nq, 16384), -7, dtype=torch.int32, device="cuda")
    H.hsa_index_full(cache, dev_bf16(q), dev(w), dev(vis), nq, T, topk, pool, ws)
    return oc, q, w, vis, cache, ws, topk, pool


@pytest.mark.parametrize("B,T,nq", FULL_CASES)
def test_index_full(hsa, B, T, nq):
    H = hsa
    oc, q, w, vis, cache, ws, topk, pool = _full_case(H, B, T, nq)
    code, flags = H.hsa_get_device_status()
    assert code == 0 and flags == 0
    topk, pool = topk.cpu().numpy(), pool.cpu().numpy()
    for b in range(B):
        K = P.dequant_index(oc, b, T)
        for i in range(nq):
            s = O.index_scores(P.f32(q[b, i]), w[b, i], K, int(vis[b, i]))
            P.check_topk(topk[b, i], s, int(vis[b, i]), name=f"topk b{b} q{i}")
            P.check_pool(pool[b, i], s, int(vis[b, i]), name=f"pool b{b} q{i}")


def test_index_full_repeatable(hsa):
    """The workspace is left clean: a second call gives the same indices."""
    H = hsa
    oc, q, w, vis, cache, ws, topk, pool = _full_case(H, 2, 9000, 1)
    t1, p1 = topk.clone(), pool.clone()
    H.hsa_index_full(cache, dev_bf16(q), dev(w), dev(vis), 1, 9000, topk, pool, ws)
    assert torch.equal(t1, topk) and torch.equal(p1, pool)


def test_index_full_ties(hsa):
    """All-equal scores (a zero query): the lowest positions and blocks win."""
    H = hsa
    T = 40000
    oc = P.oracle_cache(5, 20, 1, T, T)
    cache = gpu_cache(H, oc, T)
    q = torch.zeros(1, 1, 16, 128, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(1, 1, 16, device="cuda")
    vis = torch.tensor([[T]], dtype=torch.int32, device="cuda")
    ws = H.new_workspace(1, 1, T)
    topk = torch.empty(1, 1, 512, dtype=torch.int32, device="cuda")
    pool = torch.empty(1, 1, 16384, dtype=torch.int32, device="cuda")
    H.hsa_index_full(cache, q, w, vis, 1, T, topk, pool, ws)
    assert topk.cpu().numpy()[0, 0].tolist() == list(range(512))
    assert pool.cpu().numpy()[0, 0].tolist() == list(range(16384))


def test_index_full_wait_timeout_and_recovery(hsa):
    """Failure detection without a GPU fault: the test hook withholds one indexer-K copy of the
    Full scan, so its consumers' bounded wait (limit lowered to 2 ms) runs out. The call reports
    HSA_ERR_TIMEOUT through hsa_get_device_status, and the next call on the same workspace is
    clean and matches the oracle."""
    H = hsa
    B, T = 2, 20000
    oc, q, w, vis, cache, ws, topk, pool = _full_case(H, B, T, 1)
    code, flags = H.hsa_get_device_status()
    assert code == 0 and flags == 0
    try:
        H.hsa_set_wait_limit(2_000_000)
        H.hsa_debug_stall_next_scan()
        H.hsa_index_full(cache, dev_bf16(q), dev(w), dev(vis), 1, T, topk, pool, ws)
        code, flags = H.hsa_get_device_status()
        assert code == H.STATUS_CODES["HSA_ERR_TIMEOUT"] and flags & H.HSA_FLAG_TIMEOUT, (code, flags)
    finally:
        H.hsa_set_wait_limit(0)
    topk.fill_(-7)
    pool.fill_(-7)
    H.hsa_index_full(cache, dev_bf16(q), dev(w), dev(vis), 1, T, topk, pool, ws)
    code, flags = H.hsa_get_device_status()
    assert code == 0 and flags == 0, (code, flags)
    topk, pool = topk.cpu().numpy(), pool.cpu().numpy()
    for b in range(B):
        s = O.index_scores(P.f32(q[b, 0]), w[b, 0], P.dequant_index(oc, b, T), int(vis[b, 0]))
        P.check_topk(topk[b, 0], s, int(vis[b, 0]), name=f"after timeout topk b{b}")
        P.check_pool(pool[b, 0], s, int(vis[b, 0]), name=f"after timeout pool b{b}")


# ------------------------------------------------------------------ Reindex
@pytest.mark.parametrize("B,T,nq", [(1, 32768, 1), (2, 4100, 5), (1, 3000, 1), (1, 200000, 1), (1, 300, 1),
                                    (1, 50, 2), (1, 3000, 8)])
def test_index_reindex(hsa, B, T, nq):
    H = hsa
    oc, q, w, vis, cache, ws, topk, pool = _full_case(H, B, T, nq)
    q2 = synth.index_q_bf16(0, 24, B, nq)
    w2 = synth.index_w(0, 24, B, nq)
    out = torch.full((B, nq, 512), -7, dtype=torch.int32, device="cuda")
    H.hsa_index_reindex(cache, dev_bf16(q2), dev(w2), dev(vis), nq, T, pool, out, ws)
    code, flags = H.hsa_get_device_status()
    assert code == 0 and flags == 0
    out, pool = out.cpu().numpy(), pool.cpu().numpy()
    for b in range(B):
        K = P.dequant_index(oc, b, T)
        for i in range(nq):
            v = int(vis[b, i])
            ref, _ = O.index_reindex(P.f32(q2[b, i]), w2[b, i], K, pool[b, i], v)
            s = O.index_scores(P.f32(q2[b, i]), w2[b, i], K, v)
            g = out[b, i]
            kk = min(512, int(((pool[b, i] >= 0) & (pool[b, i] < v)).sum()))
            assert (g >= 0).sum() == kk and np.all(g[kk:] == -1) and np.all(np.diff(g[:kk]) > 0)
            assert set(g[:kk].tolist()) <= set(pool[b, i].tolist())
            P.check_set_band(g[:kk], ref[ref >= 0], s, f"reindex b{b} q{i}")
            if -(-v // 8) <= 2048:    # the pool is the whole context: reindex == full top-k
                P.check_topk(g, s, v, name="reindex-as-full")


def _reindex_direct(H, cache, q, w, T, pool_np):
    vis = torch.tensor([[T]], dtype=torch.int32, device="cuda")
    out = torch.full((1, 1, 512), -7, dtype=torch.int32, device="cuda")
    ws = H.new_workspace(1, 1, T)
    H.hsa_index_reindex(cache, q, w, vis, 1, T, dev(pool_np), out, ws)
    code, flags = H.hsa_get_device_status()
    assert code == 0 and flags == 0, (code, flags)
    return out.cpu().numpy()[0, 0]


def test_index_reindex_all_tied(hsa):
    """Every score equal (a zero query) over a pool of 2000 scattered blocks and 384 empty slots:
    each cluster CTA publishes its whole quarter (past the first half of its list) and the
    selection falls to the slot order, so the result is the pool's first 512 positions."""
    H = hsa
    T = 40000
    oc = P.oracle_cache(6, 20, 1, T, T)
    cache = gpu_cache(H, oc, T)
    blocks = np.sort(np.random.default_rng(6).choice(T // 8, 2000, replace=False))
    pool = np.full((1, 1, 16384), -1, np.int32)
    pool[0, 0, :16000] = (8 * blocks[:, None] + np.arange(8)[None, :]).reshape(-1)
    q = torch.zeros(1, 1, 16, 128, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(1, 1, 16, device="cuda")
    got = _reindex_direct(H, cache, q, w, T, pool)
    assert got.tolist() == pool[0, 0, :512].tolist()


def test_index_reindex_three_score_classes(hsa):
    """Entry e's indexer K is one of three code patterns (e % 3), so the pool's scores take three
    values and the best class is one large tie: the top-512 are that class's lowest positions,
    exactly (no tolerance band)."""
    H = hsa
    T = 20000
    rng = np.random.default_rng(7)
    pat_q = rng.integers(0, 256, (3, 64), dtype=np.uint8)
    pat_s = np.full((3, 4), 127, np.uint8)
    cls = np.arange(T) % 3
    ik_q, ik_s = pat_q[cls][None], pat_s[cls][None]
    z = np.zeros((1, T, 256), np.uint8)
    cache = H.Cache(1, T, 1, tensors=(dev(z), dev(np.zeros((1, T, 32), np.uint8)), dev(ik_q), dev(ik_s)))
    qb = synth.index_q_bf16(7, 24, 1, 1)
    wv = synth.index_w(7, 24, 1, 1)
    s3 = O.index_scores(P.f32(qb[0, 0]), wv[0, 0], O.index_k_dequant(pat_q, pat_s), 3)
    assert len(set(np.round(s3, 6).tolist())) == 3, s3
    best = int(np.argmax(s3))
    pool = np.arange(16384, dtype=np.int32)[None, None]
    got = _reindex_direct(H, cache, dev_bf16(qb), dev(wv), T, pool)
    want = np.nonzero(cls[:16384] == best)[0][:512]
    assert got.tolist() == want.tolist()


@pytest.mark.parametrize("B,T,nq", [(2, 40000, 1), (1, 16391, 1), (1, 1000, 1), (1, 200000, 2)])
def test_index_pool_tail(hsa, B, T, nq):
    """HSA_CACHE_POOL_TAIL ([ARCH] §3.3 旁路与边界): the Full call's pool gains the window blocks
    (16,544 slots per row) and the Reindex call scores them: the position top-512 is unchanged,
    the pool is checked by check_pool_tail, and Reindex over the kernel's pool against the oracle."""
    H = hsa
    cap = round8(T)
    oc = P.oracle_cache(2, 20, B, T, cap)
    q, w = synth.index_q_bf16(2, 20, B, nq), synth.index_w(2, 20, B, nq)
    q2, w2 = synth.index_q_bf16(2, 24, B, nq), synth.index_w(2, 24, B, nq)
    vis = synth.visibility(B, nq, T)
    cache = H.Cache(B, cap, 1, tensors=(dev(oc["kv_q"]), dev(oc["kv_s"]), dev(oc["ik_q"]), dev(oc["ik_s"])),
                    flags=H.HSA_CACHE_POOL_TAIL)
    ws = H.new_workspace(B, nq, T)
    n = 16384 + H.HSA_POOL_TAIL_SLOTS
    topk = torch.full((B, nq, 512), -7, dtype=torch.int32, device="cuda")
    pool = torch.full((B, nq, n), -7, dtype=torch.int32, device="cuda")
    out = torch.full((B, nq, 512), -7, dtype=torch.int32, device="cuda")
    H.hsa_index_full(cache, dev_bf16(q), dev(w), dev(vis), nq, T, topk, pool, ws)
    H.hsa_index_reindex(cache, dev_bf16(q2), dev(w2), dev(vis), nq, T, pool, out, ws)
    code, flags = H.hsa_get_device_status()
    assert code == 0 and flags == 0, (code, flags)
    topk, pool, out = topk.cpu().numpy(), pool.cpu().numpy(), out.cpu().numpy()
    for b in range(B):
        K = P.dequant_index(oc, b, T)
        for i in range(nq):
            v = int(vis[b, i])
            s = O.index_scores(P.f32(q[b, i]), w[b, i], K, v)
            P.check_topk(topk[b, i], s, v, name=f"tail topk b{b} q{i}")
            P.check_pool_tail(pool[b, i], s, v, name=f"tail pool b{b} q{i}")
            ref, _ = O.index_reindex(P.f32(q2[b, i]), w2[b, i], K, pool[b, i], v)
            s2 = O.index_scores(P.f32(q2[b, i]), w2[b, i], K, v)
            g = out[b, i]
            kk = min(512, int(((pool[b, i] >= 0) & (pool[b, i] < v)).sum()))
            assert (g >= 0).sum() == kk and np.all(g[kk:] == -1) and np.all(np.diff(g[:kk]) > 0)
            P.check_set_band(g[:kk], ref[ref >= 0], s2, f"tail reindex b{b} q{i}")


def test_index_pool_tail_window_survives(hsa):
    """The newest positions score far below every block the Full query picks, yet with the tail
    they reach the pool and a Reindex query that favours them selects them."""
    H = hsa
    T = 60000
    oc = P.oracle_cache(9, 20, 1, T, T)
    K = P.dequant_index(oc, 0, T)
    q = synth.index_q_bf16(9, 20, 1, 1)
    w = synth.index_w(9, 20, 1, 1)
    s = O.index_scores(P.f32(q[0, 0]), w[0, 0], K, T)
    m = O.block_maxima(s, T)
    blk = O.topk_ascending(m, len(m), 2048)
    assert not set(range((T - 128) // 8, T // 8)) <= set(blk.tolist())   # the plain pool misses the window
    cache = H.Cache(1, T, 1, tensors=(dev(oc["kv_q"]), dev(oc["kv_s"]), dev(oc["ik_q"]), dev(oc["ik_s"])),
                    flags=H.HSA_CACHE_POOL_TAIL)
    vis = torch.tensor([[T]], dtype=torch.int32, device="cuda")
    ws = H.new_workspace(1, 1, T)
    topk = torch.empty(1, 1, 512, dtype=torch.int32, device="cuda")
    pool = torch.empty(1, 1, 16384 + H.HSA_POOL_TAIL_SLOTS, dtype=torch.int32, device="cuda")
    H.hsa_index_full(cache, dev_bf16(q), dev(w), vis, 1, T, topk, pool, ws)
    pl = pool.cpu().numpy()[0, 0]
    assert set(range(T - 128, T)) <= set(pl.tolist())
    # a Reindex query whose heads all favour the newest entry's own direction
    qn = np.tile(np.sign(K[T - 1]).astype(np.float32), (16, 1))[None, None]
    qn_bits = (qn.view(np.uint32) >> 16).astype(np.uint16)
    wn = np.ones((1, 1, 16), np.float32)
    out = torch.empty(1, 1, 512, dtype=torch.int32, device="cuda")
    H.hsa_index_reindex(cache, dev_bf16(qn_bits), dev(wn), vis, 1, T, pool, out, ws)
    code, flags = H.hsa_get_device_status()
    assert code == 0 and flags == 0
    g = out.cpu().numpy()[0, 0]
    s2 = O.index_scores(P.f32(qn_bits[0, 0]), wn[0, 0], K, T)
    ref, _ = O.index_reindex(P.f32(qn_bits[0, 0]), wn[0, 0], K, pl, T)
    P.check_set_band(g[g >= 0], ref[ref >= 0], s2, "tail reindex, window query")
    assert T - 1 in set(g.tolist())


# ------------------------------------------------------------------ attention
def _attn_ref(oc, b, i, T, topk_row, swa_rows, q, vis, scale, fmt=O.SCALE_E8M0):
    Km = P.dequant_main(oc, b, T, fmt)
    rows = O.attention_rows(Km, topk_row, O.swa_decode(swa_rows), i, vis)
    return O.sparse_attention(P.f32(q), rows, scale)


@pytest.mark.parametrize("B,T,nq", [(1, 32768, 1), (2, 4100, 5), (1, 300, 1), (1, 50, 1), (3, 2000, 2),
                                    (1, 3000, 8)])
def test_sparse_attention(hsa, B, T, nq):
    H = hsa
    oc, q, w, vis, cache, ws, topk, pool = _full_case(H, B, T, nq)
    qa = synth.attn_q_bf16(0, 20, B, nq)
    swa = synth.swa_e4m3(0, 20, B, nq)
    out = torch.full((B, nq, 64, 512), float("nan"), device="cuda")
    H.hsa_sparse_attn_decode(cache, dev_bf16(qa), topk, dev(swa), dev(vis), nq, T, 1.0, out, ws)
    code, flags = H.hsa_get_device_status()
    assert code == 0 and flags == 0
    out, topk = out.cpu().numpy(), topk.cpu().numpy()
    for b in range(B):
        for i in range(nq):
            ref = _attn_ref(oc, b, i, T, topk[b, i], swa[b], qa[b, i], int(vis[b, i]), 1.0)
            P.check_attention(out[b, i], ref, f"attn b{b} q{i}")


def test_ragged_batch_with_empty_request(hsa):
    """Requests of 0, 5000, 37 and 1 visible positions in one batch, through the Full, Reindex
    and attention calls: the empty request gets -1 indices, an all -1 pool and a zero output;
    the others match the oracle."""
    H = hsa
    T, seed = 5000, 7
    vis_h = np.array([[0], [T], [37], [1]], np.int32)
    B, nq = vis_h.shape
    cap = round8(T)
    oc = P.oracle_cache(seed, 20, B, T, cap)
    cache = gpu_cache(H, oc, cap)
    q, w = synth.index_q_bf16(seed, 20, B, nq), synth.index_w(seed, 20, B, nq)
    q2, w2 = synth.index_q_bf16(seed, 24, B, nq), synth.index_w(seed, 24, B, nq)
    qa, swa = synth.attn_q_bf16(seed, 20, B, nq), synth.swa_e4m3(seed, 20, B, nq)
    vis = dev(vis_h)
    ws = H.new_workspace(B, nq, T)
    topk = torch.full((B, nq, 512), -7, dtype=torch.int32, device="cuda")
    pool = torch.full((B, nq, 16384), -7, dtype=torch.int32, device="cuda")
    top2 = torch.full_like(topk, -7)
    out = torch.full((B, nq, 64, 512), float("nan"), device="cuda")
    H.hsa_index_full(cache, dev_bf16(q), dev(w), vis, nq, T, topk, pool, ws)
    H.hsa_index_reindex(cache, dev_bf16(q2), dev(w2), vis, nq, T, pool, top2, ws)
    H.hsa_sparse_attn_decode(cache, dev_bf16(qa), top2, dev(swa), vis, nq, T, 1.0, out, ws)
    code, flags = H.hsa_get_device_status()
    assert code == 0 and flags == 0, (code, flags)
    topk, pool, top2, out = topk.cpu().numpy(), pool.cpu().numpy(), top2.cpu().numpy(), out.cpu().numpy()
    assert np.all(topk[0] == -1) and np.all(pool[0] == -1) and np.all(top2[0] == -1) and np.all(out[0] == 0)
    for b in range(B):
        v = int(vis_h[b, 0])
        K = P.dequant_index(oc, b, T)
        s = O.index_scores(P.f32(q[b, 0]), w[b, 0], K, v)
        P.check_topk(topk[b, 0], s, v, name=f"ragged topk b{b}")
        P.check_pool(pool[b, 0], s, v, name=f"ragged pool b{b}")
        ref2, _ = O.index_reindex(P.f32(q2[b, 0]), w2[b, 0], K, pool[b, 0], v)
        s2 = O.index_scores(P.f32(q2[b, 0]), w2[b, 0], K, v)
        assert np.sum(top2[b, 0] >= 0) == np.sum(ref2 >= 0), f"ragged reindex b{b}: count"
        if v > 0:
            P.check_set_band(top2[b, 0][top2[b, 0] >= 0], ref2[ref2 >= 0], s2, f"ragged reindex b{b}")
        ref = _attn_ref(oc, b, 0, T, top2[b, 0], swa[b], qa[b, 0], v, 1.0)
        P.check_attention(out[b, 0], ref, f"ragged attn b{b}")


def test_sparse_attention_scale_and_e4m3_scales(hsa):
    H = hsa
    T, fmt = 6000, O.SCALE_E4M3
    oc = P.oracle_cache(3, 20, 1, T, T, scale_fmt=fmt)
    cache = gpu_cache(H, oc, T, fmt)
    rng = np.random.default_rng(0)
    topk = np.sort(rng.choice(T, 512, replace=False)).astype(np.int32)[None, None]
    qa = synth.attn_q_bf16(3, 21, 1, 1)
    swa = synth.swa_e4m3(3, 21, 1, 1)
    vis = np.array([[T]], np.int32)
    out = torch.empty(1, 1, 64, 512, device="cuda")
    ws = H.new_workspace(1, 1, T)
    H.hsa_sparse_attn_decode(cache, dev_bf16(qa), dev(topk), dev(swa), dev(vis), 1, T, 3.0, out, ws)
    ref = _attn_ref(oc, 0, 0, T, topk[0, 0], swa[0], qa[0, 0], T, 3.0, fmt)
    P.check_attention(out.cpu().numpy()[0, 0], ref, "attn e4m3 scale 3")


def test_sparse_attention_flags_bad_index(hsa):
    H = hsa
    T = 1000
    oc = P.oracle_cache(4, 20, 1, T, T)
    cache = gpu_cache(H, oc, T)
    topk = np.full((1, 1, 512), -1, np.int32)
    topk[0, 0, :3] = [5, 999, 1200]          # 1200 >= vis: skipped and flagged
    qa = synth.attn_q_bf16(4, 20, 1, 1)
    swa = synth.swa_e4m3(4, 20, 1, 1)
    out = torch.empty(1, 1, 64, 512, device="cuda")
    ws = H.new_workspace(1, 1, T)
    H.hsa_sparse_attn_decode(cache, dev_bf16(qa), dev(topk), dev(swa), dev(np.array([[T]], np.int32)), 1, T, 1.0,
                             out, ws)
    code, flags = H.hsa_get_device_status()
    assert flags & H.HSA_FLAG_INDEX_RANGE
    ref = _attn_ref(oc, 0, 0, T, np.array([5, 999]), swa[0], qa[0, 0], T, 1.0)
    P.check_attention(out.cpu().numpy()[0, 0], ref, "attn bad index")


# ------------------------------------------------------------------ schedule
def test_schedule_step(hsa):
    """Each layer slot owns its cache: the Full slot scores layer 20's indexer K, the Reindex slot
    rescores the pool over layer 24's, and every slot attends over its own main KV."""
    H = hsa
    B, T, nq, seed = 2, 12345, 1, 0
    layers = [20, 21, 24, 25]
    modes = [H.HSA_MODE_FULL, H.HSA_MODE_REUSE, H.HSA_MODE_REINDEX, H.HSA_MODE_REUSE]
    cap = round8(T)
    oc = {l: P.oracle_cache(seed, l, B, T, cap) for l in layers}
    caches = [gpu_cache(H, oc[l], cap) for l in layers]
    vis = synth.visibility(B, nq, T)
    qi = {l: synth.index_q_bf16(seed, l, B, nq) for l in (20, 24)}
    wi = {l: synth.index_w(seed, l, B, nq) for l in (20, 24)}
    qa = {l: synth.attn_q_bf16(seed, l, B, nq) for l in layers}
    sw = {l: synth.swa_e4m3(seed, l, B, nq) for l in layers}
    d_qi = [dev_bf16(qi[l]) if l in qi else None for l in layers]
    d_wi = [dev(wi[l]) if l in wi else None for l in layers]
    d_qa = [dev_bf16(qa[l]) for l in layers]
    d_sw = [dev(sw[l]) for l in layers]
    outs = [torch.empty(B, nq, 64, 512, device="cuda") for _ in layers]
    tk = [torch.empty(B, nq, 512, dtype=torch.int32, device="cuda") if l in qi else None for l in layers]
    pool = torch.empty(B, nq, 16384, dtype=torch.int32, device="cuda")
    d_vis = dev(vis)
    ws = H.new_workspace(B, nq, T)
    step = H.StepArgs(modes, d_qi, d_wi, d_qa, d_sw, outs, tk, pool, d_vis, nq, T, 1.0)
    H.hsa_schedule_step(caches, step, ws)
    code, flags = H.hsa_get_device_status()
    assert code == 0 and flags == 0
    pool_h = pool.cpu().numpy()
    t20, t24 = tk[0].cpu().numpy(), tk[2].cpu().numpy()
    for b in range(B):
        K20, K24 = P.dequant_index(oc[20], b, T), P.dequant_index(oc[24], b, T)
        s20 = O.index_scores(P.f32(qi[20][b, 0]), wi[20][b, 0], K20, T)
        P.check_topk(t20[b, 0], s20, T, name="step L20")
        P.check_pool(pool_h[b, 0], s20, T, name="step pool")
        ref24, _ = O.index_reindex(P.f32(qi[24][b, 0]), wi[24][b, 0], K24, pool_h[b, 0], T)
        s24 = O.index_scores(P.f32(qi[24][b, 0]), wi[24][b, 0], K24, T)
        P.check_set_band(t24[b, 0][t24[b, 0] >= 0], ref24[ref24 >= 0], s24, "step L24")
        for j, l in enumerate(layers):
            idx = t20 if l < 24 else t24
            ref = _attn_ref(oc[l], b, 0, T, idx[b, 0], sw[l][b], qa[l][b, 0], T, 1.0)
            P.check_attention(outs[j].cpu().numpy()[b, 0], ref, f"step attn L{l}")


def test_chained_calls_read_fresh_outputs(hsa):
    """Every call is launched with programmatic dependent launch: a kernel starts while its
    predecessor may still run, and must read what the predecessor writes (cache rows, the pool,
    a top-k) only after its dependency wait and through coherent loads. Before each chained
    round, every index buffer is filled with the other query's valid, different result (plain
    copies, which complete before the chain starts), so a read that overtakes its producer
    returns another in-range index set; the latent sets alternate, so an early row read returns
    other rows. Each reader directly follows its producer: cache write -> attention, Full ->
    Reindex (pool), Reindex -> attention (top-k), Full -> attention (top-k); then the same work
    as one schedule_step. Every round must equal the same calls separated by synchronisations,
    bit for bit, with no device flag. Batch 16 at 65,536 positions keeps each producer running
    long enough for an early read to land before its writes."""
    H = hsa
    B, T, nq = 16, 65536, 1
    torch.manual_seed(11)
    W = (torch.randn(512, 128, device="cuda") / 22.6).to(torch.bfloat16)
    lat = [torch.randn(B, T, 512, device="cuda").to(torch.bfloat16) for _ in range(2)]
    qi = [torch.randn(B, nq, 16, 128, device="cuda").to(torch.bfloat16) for _ in range(2)]
    wi = torch.rand(B, nq, 16, device="cuda")
    qi2 = torch.randn(B, nq, 16, 128, device="cuda").to(torch.bfloat16)
    qa = (torch.randn(B, nq, 64, 512, device="cuda") / 22.6).to(torch.bfloat16)
    swa = torch.randn(B, 128 + nq - 1, 512, device="cuda").to(torch.float8_e4m3fn).view(torch.uint8)
    vis = torch.full((B, nq), T, dtype=torch.int32, device="cuda")
    fixed = torch.randint(0, T, (B, nq, 512), dtype=torch.int32, device="cuda")
    cache = H.Cache(B, T, 1)
    ws = H.new_workspace(B, nq, T)
    topk = torch.empty(B, nq, 512, dtype=torch.int32, device="cuda")
    top2 = torch.empty_like(topk)
    pool = torch.empty(B, nq, 16384, dtype=torch.int32, device="cuda")
    out = [torch.empty(B, nq, 64, 512, device="cuda") for _ in range(3)]

    def flags_clear(tag):
        code, flags = H.hsa_get_device_status()
        assert code == 0 and flags == 0, (tag, code, flags)

    def calls(c, q, sync, stale=None):
        fence = torch.cuda.synchronize if sync else (lambda: None)
        if stale is not None:
            topk.copy_(stale[1])
            pool.copy_(stale[2])
            top2.copy_(stale[3])
        H.hsa_cache_write_compress(cache, lat[c], None, W, T, None)
        fence()
        H.hsa_sparse_attn_decode(cache, qa, fixed, swa, vis, nq, T, 1.0, out[0], ws)
        fence()
        H.hsa_index_full(cache, qi[q], wi, vis, nq, T, topk, pool, ws)
        fence()
        H.hsa_index_reindex(cache, qi2, wi, vis, nq, T, pool, top2, ws)
        fence()
        H.hsa_sparse_attn_decode(cache, qa, top2, swa, vis, nq, T, 1.0, out[1], ws)
        torch.cuda.synchronize()
        res = [out[0].clone(), topk.clone(), pool.clone(), top2.clone(), out[1].clone()]
        if stale is not None:
            topk.copy_(stale[1])
        H.hsa_index_full(cache, qi[q], wi, vis, nq, T, topk, pool, ws)
        fence()
        H.hsa_sparse_attn_decode(cache, qa, topk, swa, vis, nq, T, 1.0, out[2], ws)
        torch.cuda.synchronize()
        flags_clear(("calls", c, q, sync))
        return res + [out[2].clone()]

    modes = [H.HSA_MODE_FULL, H.HSA_MODE_REUSE, H.HSA_MODE_REINDEX, H.HSA_MODE_REUSE]
    s_out = [torch.empty_like(out[0]) for _ in modes]
    s_tk = [torch.empty_like(topk), None, torch.empty_like(topk), None]
    s_pool = torch.empty_like(pool)
    q_step = torch.empty_like(qi[0])
    step = H.StepArgs(modes, [q_step, None, qi2, None], [wi, None, wi, None], [qa] * 4, [swa] * 4, s_out, s_tk,
                      s_pool, vis, nq, T, 1.0)

    def stepped(c, q, stale):
        s_tk[0].copy_(stale[1])
        s_pool.copy_(stale[2])
        s_tk[2].copy_(stale[3])
        q_step.copy_(qi[q])
        H.hsa_cache_write_compress(cache, lat[c], None, W, T, None)
        H.hsa_schedule_step(cache, step, ws)
        torch.cuda.synchronize()
        flags_clear(("step", c, q))
        return [s_tk[0].clone(), s_pool.clone(), s_out[0].clone(), s_out[1].clone(), s_tk[2].clone(),
                s_out[2].clone(), s_out[3].clone()]

    ref = {(c, q): calls(c, q, True) for c in (0, 1) for q in (0, 1)}
    # the queries give different index sets and the latent sets different rows, else the
    # rounds would show nothing
    assert not torch.equal(ref[(0, 0)][2], ref[(0, 1)][2]) and not torch.equal(ref[(0, 0)][3], ref[(0, 1)][3])
    assert not torch.equal(ref[(0, 0)][0], ref[(1, 0)][0])
    names = ("attention after the cache write", "Full top-k", "pool", "Reindex top-k",
             "attention on the Reindex top-k", "attention on the Full top-k")
    slots = ("Full top-k", "pool", "Full slot output", "Reuse slot output", "Reindex top-k",
             "Reindex slot output", "second Reuse slot output")
    for c, q in [(0, 0), (1, 1), (0, 1), (1, 0)] * 2:
        want = ref[(c, q)]
        stale = ref[(c, 1 - q)]
        for name, x, y in zip(names, calls(c, q, False, stale), want):
            assert torch.equal(x, y), f"chained calls, latents {c}, query {q}: {name} differs"
        o0, tk_r, pool_r, t2_r, o2_r, o1_r = want
        for name, x, y in zip(slots, stepped(c, q, stale), (tk_r, pool_r, o1_r, o1_r, t2_r, o2_r, o2_r)):
            assert torch.equal(x, y), f"schedule_step, latents {c}, query {q}: {name} differs"


def test_schedule_step_matches_standalone_calls(hsa):
    """Inside hsa_schedule_step the kernels read step inputs before their dependency wait and a
    Reindex or Reuse-slot attention kernel waits only before its first global write; the
    arithmetic is that of the standalone calls, so the step's indices and outputs equal theirs
    bit for bit (two requests, a ragged length, slots Full, Reuse, Reindex, Reuse, Reuse, each
    slot over its own layer's cache)."""
    H = hsa
    B, T, nq, seed = 2, 12345, 1, 3
    layers = [20, 21, 24, 25, 26]
    modes = [H.HSA_MODE_FULL, H.HSA_MODE_REUSE, H.HSA_MODE_REINDEX, H.HSA_MODE_REUSE, H.HSA_MODE_REUSE]
    cap = round8(T)
    cache = {l: gpu_cache(H, P.oracle_cache(seed, l, B, T, cap), cap) for l in layers}
    d_vis = dev(synth.visibility(B, nq, T))
    d_qi = {l: dev_bf16(synth.index_q_bf16(seed, l, B, nq)) for l in (20, 24)}
    d_wi = {l: dev(synth.index_w(seed, l, B, nq)) for l in (20, 24)}
    d_qa = {l: dev_bf16(synth.attn_q_bf16(seed, l, B, nq)) for l in layers}
    d_sw = {l: dev(synth.swa_e4m3(seed, l, B, nq)) for l in layers}
    ws = H.new_workspace(B, nq, T)
    new_idx = lambda: torch.empty(B, nq, 512, dtype=torch.int32, device="cuda")  # noqa: E731
    new_out = lambda: torch.empty(B, nq, 64, 512, device="cuda")  # noqa: E731

    # standalone calls, one after the other
    t20, pool, t24 = new_idx(), torch.empty(B, nq, 16384, dtype=torch.int32, device="cuda"), new_idx()
    H.hsa_index_full(cache[20], d_qi[20], d_wi[20], d_vis, nq, T, t20, pool, ws)
    H.hsa_index_reindex(cache[24], d_qi[24], d_wi[24], d_vis, nq, T, pool, t24, ws)
    ref = {}
    for l in layers:
        ref[l] = new_out()
        H.hsa_sparse_attn_decode(cache[l], d_qa[l], t20 if l < 24 else t24, d_sw[l], d_vis, nq, T, 1.0, ref[l], ws)

    # the same work as one step
    outs = [new_out() for _ in layers]
    tk = [new_idx() if l in d_qi else None for l in layers]
    s_pool = torch.empty_like(pool)
    step = H.StepArgs(modes, [d_qi.get(l) for l in layers], [d_wi.get(l) for l in layers],
                      [d_qa[l] for l in layers], [d_sw[l] for l in layers], outs, tk, s_pool, d_vis, nq, T, 1.0)
    H.hsa_schedule_step([cache[l] for l in layers], step, ws)
    code, flags = H.hsa_get_device_status()
    assert code == 0 and flags == 0
    assert torch.equal(tk[0], t20) and torch.equal(s_pool, pool) and torch.equal(tk[2], t24)
    for j, l in enumerate(layers):
        assert torch.equal(outs[j], ref[l]), f"slot {j} (layer {l})"
