"""Pins for the fp64 oracle: closed forms and worked examples printed on the pages, library
routines, brute force on tiny inputs, and invariants the method implies. None of these
re-runs the oracle's own formula. Each test is built so that a plausible slip in the oracle
fails it: a dropped term, a wrong sign or index, or a swapped operand or nibble."""
import math

import numpy as np
import pytest
import torch

import oracle as O
from hierarchical_sparse_attention_index_gb300 import synth
from tests.conftest import read_golden


# ------------------------------------------------------------------ number formats
def test_e4m3_decode_matches_torch_float8():
    b = torch.arange(256, dtype=torch.uint8)
    ref = b.view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    got = O.e4m3_decode(np.arange(256))
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    m = ~np.isnan(ref)
    assert np.array_equal(ref[m], got[m])
    # the pages' maximum: 448 ([ARCH] §7, 448 x 6 = 2688)
    assert np.nanmax(got) == 448.0


def test_e8m0_decode_matches_torch_float8():
    b = torch.arange(256, dtype=torch.uint8)
    ref = b.view(torch.float8_e8m0fnu).float().numpy().astype(np.float64)
    got = O.e8m0_decode(np.arange(256))
    assert np.isnan(got[255]) and np.isnan(ref[255])
    # torch's float32 cannot hold 2^-127 exactly as a normal but does as a subnormal
    assert np.array_equal(ref[:255], got[:255])


def test_e2m1_table_and_page_maximum():
    rows = read_golden("e2m1_table.txt")
    for nib, val in rows:
        v = O.e2m1_decode(int(nib))
        assert v == float(val)
        assert math.copysign(1.0, v) == math.copysign(1.0, float(val)) or float(val) == 0.0
    vals = O.e2m1_decode(np.arange(16))
    # 448 x 6 = 2688 is the format's maximum magnitude ([ARCH] §7)
    assert float(np.max(vals)) * float(np.nanmax(O.e4m3_decode(np.arange(256)))) == 2688.0
    # 16 code points, 15 distinct values ("FP4 只有 16 个可表示值", +0 and -0 coincide)
    assert len(set(vals.tolist())) == 15


def _brute_nearest_even(v):
    """Brute force: nearest of the 8 magnitudes; on a tie the code with mantissa bit 0."""
    mags = O.e2m1_decode(np.arange(8))
    a = abs(float(np.float32(v)))
    if a > 6.0:
        code = 7
    else:
        d = np.abs(mags - a)
        best = np.nonzero(d == d.min())[0]
        code = int(best[0]) if len(best) == 1 else int([c for c in best if (c & 1) == 0][0])
    if code != 0 and v < 0:
        code |= 8
    return code


def test_e2m1_encode_brute_force_round_to_nearest_even():
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    pts = []
    for m in mids:
        pts += [m, np.nextafter(np.float32(m), np.float32(0)), np.nextafter(np.float32(m), np.float32(9))]
    pts += list(O.e2m1_decode(np.arange(8)))
    pts += [6.0, 6.5, 100.0, 1e-30, 0.0]
    rng = np.random.default_rng(1)
    pts += list(rng.uniform(0, 7, 4000))
    pts = np.array(pts, dtype=np.float32)
    pts = np.concatenate([pts, -pts])
    got = O.e2m1_encode(pts)
    ref = np.array([_brute_nearest_even(v) for v in pts], dtype=np.uint8)
    assert np.array_equal(got, ref)
    # -0 never stored: a tiny negative rounds to code 0, not 8
    assert O.e2m1_encode(np.float32(-0.1)) == 0


def test_scale_rules_brute_force():
    rng = np.random.default_rng(2)
    amax = np.concatenate([rng.lognormal(0, 3, 3000), [0.0, 6.0, 3.0, 12.0, 6 * 2.0 ** -10,
                                                       np.nextafter(6.0, 7.0), 1e-40, 448 * 6, 1e6]])
    e8 = O.e8m0_decode(np.arange(255))
    e4 = O.e4m3_decode(np.arange(1, 127))
    for a in amax:
        b = int(O.e8m0_scale_byte(a))
        ok = np.nonzero(6.0 * e8 >= a)[0]
        want = 0 if a == 0 else int(ok[0])
        assert b == want, (a, b, want)
        b4 = int(O.e4m3_scale_byte(a))
        ok4 = np.nonzero(6.0 * e4 >= a)[0]
        want4 = (int(ok4[0]) + 1) if len(ok4) else 126
        assert b4 == want4, (a, b4, want4)


@pytest.mark.parametrize("fmt", [O.SCALE_E8M0, O.SCALE_E4M3])
@pytest.mark.parametrize("group", [16, 32])
def test_quantise_bounds_and_roundtrip(fmt, group):
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((200, 128)) * rng.lognormal(0, 2, (200, 1))).astype(np.float32)
    if fmt == O.SCALE_E4M3:          # keep amax under 6 x 448, where the E4M3 scale saturates
        x = np.clip(x, -2000, 2000)
    x[0] = 0.0
    q, s = O.quantise_groups(x, group, fmt)
    assert q.shape == (200, 64) and s.shape == (200, 128 // group)
    deq = O.dequant_groups(q, s, group, fmt)
    sc = (O.e8m0_decode(s) if fmt == O.SCALE_E8M0 else O.e4m3_decode(s))
    g = x.reshape(200, -1, group).astype(np.float64)
    # |x / s| <= 6 and the error is at most half of the widest grid step (1.0) times s
    assert np.all(np.abs(g) <= 6 * sc[:, :, None] * (1 + 1e-7))
    assert np.all(np.abs(deq.reshape(g.shape) - g) <= 1.0 * sc[:, :, None] + 1e-30)
    # E8M0: re-quantising a dequantised group reproduces it exactly (amax/s lands on 4 or 6,
    # so the power-of-two scale is chosen again and every value is a grid point)
    if fmt == O.SCALE_E8M0:
        q2, s2 = O.quantise_groups(deq.astype(np.float32), group, fmt)
        assert np.array_equal(O.dequant_groups(q2, s2, group, fmt), deq)
    assert np.all(deq[0] == 0)


def test_index_k_fragment_order():
    for stored, t, s_, i, lo, hi in read_golden("index_k_fragment_order.txt"):
        stored = int(stored)
        assert stored == 16 * int(t) + 2 * int(s_) + int(i)
        row = np.zeros((1, 64), np.uint8)
        row[0, stored] = 0x21                      # low nibble 1 (+0.5), high nibble 2 (+1.0)
        vals = O.index_k_dequant(row, np.full((1, 4), 127, np.uint8))[0]
        nz = np.nonzero(vals)[0].tolist()
        assert nz == [int(lo), int(hi)] and vals[int(lo)] == 0.5 and vals[int(hi)] == 1.0
    # the stored order is a permutation: natural -> stored -> natural is the identity
    rng = np.random.default_rng(0)
    x = rng.integers(0, 256, (5, 64)).astype(np.uint8)
    assert np.array_equal(O.index_k_to_natural(O.index_k_to_stored(x)), x)


def test_nibble_order_low_first():
    x = np.zeros((1, 32), np.float32)
    x[0, 0] = 6.0     # element 0 -> low nibble of byte 0
    x[0, 1] = -1.0    # element 1 -> high nibble of byte 0
    q, s = O.quantise_groups(x, 32, O.SCALE_E8M0)
    assert s[0, 0] == 127
    assert q[0, 0] == (0x7 | (0xA << 4))


# ------------------------------------------------------------------ byte accounting
def test_byte_counts_from_pages():
    g = {k: float(v) for k, v in read_golden("byte_counts.txt")}
    main, idx = O.entry_bytes()
    assert main == g["main_kv_slot"] and idx == g["index_k_slot"]
    assert main + idx == g["slot_total"]
    assert (main + idx) / 2 == g["per_token_ratio2"] and (main + idx) / 1 == g["per_token_ratio1"]
    ratios = [O.compress_ratios()[layer] for layer in O.KV_SOURCE_LAYERS]
    assert O.global_kv_bytes_per_token(ratios) == g["global_per_token"]
    reindex_layers = [lay for lay in O.INDEX_SOURCE_LAYERS if lay not in O.KV_SOURCE_LAYERS]
    assert O.global_kv_bytes_per_token(ratios, reindex_layers) == g["wrong_count_with_reindex_k"]
    assert O.global_kv_bytes_per_token(ratios) * (1 << 20) / (1 << 20) == g["mib_per_1m_tokens"]


# ------------------------------------------------------------------ schedule
def test_layer_schedule_matches_page_table():
    modes = O.layer_modes()
    ratios = O.compress_ratios()
    assert len(modes) == 43 and len(ratios) == 43
    for first, last, ratio, mode in read_golden("layer_schedule.txt"):
        for layer in range(int(first), int(last) + 1):
            assert modes[layer] == mode, layer
            assert ratios[layer] == int(ratio), layer


def test_decoder_step_counts():
    assert O.decoder_step_counts() == (1, 4, 15)
    producers = [i for i, m in enumerate(O.layer_modes()) if m in ("Full", "Reindex") and i >= 20]
    assert producers == [20, 24, 28, 32, 36]
    # K storage exists only on the four KV sources
    assert [i for i, m in enumerate(O.layer_modes()) if m == "Full"] == [2, 8, 14, 20]


# ------------------------------------------------------------------ indexer score
def test_score_worked_example():
    q = np.zeros((16, 128))
    q[0, 0] = 2.0
    q[1, 1] = -1.0
    q[2, 0] = q[2, 1] = q[2, 32] = 1.0
    w = np.zeros(16)
    w[:3] = [0.5, 0.25, 1.0]
    rows = read_golden("score_worked_example.txt")
    ik_q = np.zeros((len(rows), 64), np.uint8)
    ik_s = np.zeros((len(rows), 4), np.uint8)
    want = []
    for i, (_, b0, b16, s0, s1, s2, s3, exp) in enumerate(rows):
        ik_q[i, 0] = int(b0, 16)
        ik_q[i, 4] = int(b16, 16)
        ik_s[i] = [int(s0), int(s1), int(s2), int(s3)]
        want.append(float(exp))
    K = O.index_k_dequant(ik_q, ik_s)
    s = O.index_scores(q, w, K, len(rows))
    assert np.array_equal(s, np.array(want))


def test_score_special_cases():
    rng = np.random.default_rng(4)
    q = rng.standard_normal((16, 128))
    K = rng.standard_normal((50, 128))
    for h in (0, 7, 15):
        w = np.zeros(16)
        w[h] = 1.0
        s = O.index_scores(q, w, K, 50)
        ref = np.array([max(0.0, float(np.dot(q[h], K[t]))) for t in range(50)])
        np.testing.assert_allclose(s, ref, rtol=1e-12, atol=1e-12)
    # positions at or beyond vis are never scored
    s = O.index_scores(q, np.ones(16), K, 20)
    assert np.all(np.isneginf(s[20:])) and np.all(np.isfinite(s[:20]))
    # negating every query makes each dot change sign: the ReLU terms swap roles
    w = rng.random(16)
    sp = O.index_scores(q, w, K, 50)
    sn = O.index_scores(-q, w, K, 50)
    dots = K @ q.T
    np.testing.assert_allclose(sp - sn, dots @ w, rtol=1e-10, atol=1e-9)


# ------------------------------------------------------------------ top-k, blocks, pool
def _brute_topk(s, n, k):
    items = sorted(range(n), key=lambda t: (-float(np.float32(s[t])), t))
    return sorted(items[:min(k, n)])


@pytest.mark.parametrize("T", [1, 7, 8, 9, 511, 512, 513, 1000])
def test_topk_brute_force(T):
    rng = np.random.default_rng(T)
    s = rng.standard_normal(T)
    s[rng.integers(0, T, T // 3)] = 0.5          # plant exact ties
    for k in (1, 5, 512):
        got = O.topk_ascending(s, T, k)
        assert got.tolist() == _brute_topk(s, T, k)


def test_block_maxima_and_pool_brute_force():
    rng = np.random.default_rng(5)
    for vis in (1, 7, 8, 9, 100, 16383, 16384, 16385, 40000):
        s = rng.standard_normal(vis + 5)
        m = O.block_maxima(s, vis)
        assert len(m) == math.ceil(vis / 8)
        for b in range(len(m)):
            assert m[b] == max(s[8 * b:min(vis, 8 * b + 8)])
        blk = O.topk_ascending(m, len(m), 2048)
        pool = O.expand_pool(blk, vis)
        live = pool[:len(blk) * 8]
        assert len(blk) * 8 == O.pool_size(vis)
        assert np.all(pool[len(blk) * 8:] == -1)
        assert all((p == -1) or (p < vis) for p in live)
        if math.ceil(vis / 8) <= 2048:
            assert sorted(p for p in live if p >= 0) == list(range(vis))


def test_pool_size_closed_form():
    for T, want in [(1, 8), (7, 8), (8, 8), (9, 16), (16383, 16384), (16384, 16384),
                    (16385, 16384), (131072, 16384), (1 << 20, 16384), (0, 0)]:
        assert O.pool_size(T) == want
    assert O.POOL_SLOTS == 16384 == 2048 * 8


def test_full_topk_inside_pool_block_max_is_upper_bound():
    rng = np.random.default_rng(6)
    q = synth.bf16_bits_to_f32(synth.index_q_bf16(7, 20, 1, 1))[0, 0].astype(np.float64)
    w = rng.random(16)
    for T in (20000, 50000):
        K = rng.standard_normal((T, 128))
        topk, pool, s, m = O.index_full(q, w, K, T)
        assert set(topk.tolist()) <= set(pool[pool >= 0].tolist())


def test_full_topk_inside_top512_blocks_with_ties():
    """The position top-512 lies inside the 8-position blocks ranked in the top 512 by block max
    ([ARCH] §3.3: the block max is an upper bound), with both orders breaking ties towards the
    lower index. Scores drawn from a few integers force ties at every level."""
    rng = np.random.default_rng(61)
    for T in (4100, 9001, 40000):
        for levels in (3, 7, 1000):
            s = rng.integers(0, levels, T).astype(np.float64)
            top = O.topk_ascending(s, T, 512)
            m = O.block_maxima(s, T)
            blocks = O.topk_ascending(m, len(m), 512)
            inside = set((blocks[:, None] * 8 + np.arange(8)[None, :]).ravel().tolist())
            assert set(top.tolist()) <= inside, (T, levels)
            # and the 512th block max never exceeds the 512th position score
            assert m[blocks].min() <= s[top].min()


def test_reindex_over_whole_context_equals_full():
    rng = np.random.default_rng(8)
    T = 12000                                   # ceil(T/8) <= 2048: the pool is everything
    K = rng.standard_normal((T, 128))
    q1, q2 = rng.standard_normal((2, 16, 128))
    w1, w2 = rng.random((2, 16))
    _, pool, _, _ = O.index_full(q1, w1, K, T)
    re, _ = O.index_reindex(q2, w2, K, pool, T)
    full2, _, _, _ = O.index_full(q2, w2, K, T)
    assert np.array_equal(re, full2)


def test_short_context_takes_everything():
    rng = np.random.default_rng(9)
    K = rng.standard_normal((300, 128))
    topk, pool, _, _ = O.index_full(rng.standard_normal((16, 128)), rng.random(16), K, 300)
    assert topk[:300].tolist() == list(range(300)) and np.all(topk[300:] == -1)
    assert pool[:300].tolist() == list(range(300)) and np.all(pool[300:] == -1)


def test_planted_clusters_are_selected():
    seed, T = 77, 65536
    lat = synth.latents_bf16(seed, 20, 0, T)
    W = synth.w_idx_bf16(seed, 20)
    qb = synth.index_q_bf16(seed, 20, 1, 1)[0, 0]
    w = synth.index_w(seed, 20, 1, 1)[0, 0]
    planted = synth.plant_clusters(lat, W, qb, w, 64, seed, 0)
    wkv = synth.bf16_bits_to_f32(lat)
    _, _, ik_q, ik_s, _, _ = O.cache_write_compress(wkv, None, synth.bf16_bits_to_f32(W), 1)
    K = O.index_k_dequant(ik_q, ik_s)
    topk, pool, s, _ = O.index_full(synth.bf16_bits_to_f32(qb), w, K, T)
    assert topk.tolist() == sorted(planted.tolist())
    assert set(planted.tolist()) <= set(pool.tolist())
    others = np.delete(s, planted)
    assert s[planted].min() >= 2.0 * others.max()


# ------------------------------------------------------------------ attention
def test_attention_special_cases():
    rng = np.random.default_rng(10)
    q = rng.standard_normal((64, 512)) * 0.05
    rows = rng.standard_normal((37, 512))
    # one key: every head returns it
    o = O.sparse_attention(q, rows[:1], 1.0)
    assert np.allclose(o, np.broadcast_to(rows[0], o.shape), rtol=0, atol=1e-12)
    # zero query (or zero scale): the plain mean of the keys
    o = O.sparse_attention(np.zeros_like(q), rows, 1.0)
    np.testing.assert_allclose(o, np.broadcast_to(rows.mean(0), o.shape), rtol=1e-12, atol=1e-12)
    # row order is irrelevant
    perm = rng.permutation(37)
    np.testing.assert_allclose(O.sparse_attention(q, rows, 0.7), O.sparse_attention(q, rows[perm], 0.7),
                               rtol=1e-12, atol=1e-12)
    # against scipy's softmax (a library routine), large logits included
    from scipy.special import softmax
    for scale in (0.3, 40.0):
        ref = softmax(scale * (q @ rows.T), axis=1) @ rows
        np.testing.assert_allclose(O.sparse_attention(q, rows, scale), ref, rtol=1e-10, atol=1e-12)


def test_attention_two_key_worked_example():
    # logits a1 = 0, a2 = ln 3 -> weights 1/4, 3/4
    k1 = np.zeros(512)
    k1[0] = 4.0
    k2 = np.zeros(512)
    k2[1] = 8.0
    q = np.zeros((64, 512))
    q[:, 1] = math.log(3.0) / 8.0
    o = O.sparse_attention(q, np.stack([k1, k2]), 1.0)
    assert np.allclose(o[:, 0], 1.0) and np.allclose(o[:, 1], 6.0)


def test_attention_rows_mapping():
    Km = np.arange(20 * 512, dtype=np.float64).reshape(20, 512)
    swa = -np.arange((128 + 2) * 512, dtype=np.float64).reshape(130, 512)
    topk = np.array([3, 7, -1, 11] + [-1] * 508)
    # long context: 3 valid top-k rows + the full window [q_index, q_index + 128)
    rows = O.attention_rows(Km, topk, swa, 2, 1000)
    assert rows.shape[0] == 3 + 128
    assert np.array_equal(rows[:3], Km[[3, 7, 11]]) and np.array_equal(rows[3:], swa[2:130])
    # vis = 12 < W: only the last 12 window rows hold real positions; index 11 is visible
    rows = O.attention_rows(Km, topk, swa, 0, 12)
    assert rows.shape[0] == 3 + 12 and np.array_equal(rows[3:], swa[116:128])
    rows = O.attention_rows(Km, topk, swa, 0, 10)   # index 11 not visible
    assert rows.shape[0] == 2 + 10


# ------------------------------------------------------------------ compressor
def test_compressor_pooling_special_cases():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((6, 512))
    # equal gates: the plain mean of the pair
    p = O.compress_pool(x, np.zeros((6, 512)), 2)
    np.testing.assert_allclose(p, 0.5 * (x[0::2] + x[1::2]), rtol=1e-12, atol=1e-12)
    # a gate gap of 50 picks the token with the larger gate, channel by channel
    g = np.zeros((6, 512))
    g[0::2, :256] = 50.0
    g[1::2, 256:] = 50.0
    p = O.compress_pool(x, g, 2)
    np.testing.assert_allclose(p[:, :256], x[0::2, :256], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(p[:, 256:], x[1::2, 256:], rtol=1e-12, atol=1e-12)
    # odd tail not written; m = 1 is the identity
    assert O.compress_pool(x[:5], g[:5], 2).shape == (2, 512)
    assert np.array_equal(O.compress_pool(x, None, 1), x)


def test_rms_norm_unit_rms():
    rng = np.random.default_rng(12)
    x = rng.standard_normal((10, 512)) * rng.lognormal(0, 2, (10, 1))
    y = O.rms_norm(x)
    ms = np.mean(x * x, axis=1)
    np.testing.assert_allclose(np.mean(y * y, axis=1), ms / (ms + O.RMS_EPS), rtol=1e-12)
    # direction kept
    np.testing.assert_allclose(y / np.linalg.norm(y, axis=1, keepdims=True),
                               x / np.linalg.norm(x, axis=1, keepdims=True), rtol=1e-12, atol=1e-15)


def test_cache_write_projection_selects_channels():
    rng = np.random.default_rng(13)
    wkv = rng.standard_normal((8, 512))
    W = np.zeros((512, 128))
    W[np.arange(128) + 100, np.arange(128)] = 1.0         # K = latent[:, 100:228]
    kv_q, kv_s, ik_q, ik_s, lat, K = O.cache_write_compress(wkv, None, W, 1)
    assert np.array_equal(K, lat[:, 100:228])
    # the m = 1 entry is the normalised projection, quantised
    np.testing.assert_allclose(lat, O.rms_norm(wkv), rtol=0, atol=0)
    assert kv_q.shape == (8, 256) and kv_s.shape == (8, 32) and ik_q.shape == (8, 64) and ik_s.shape == (8, 4)


def test_decode_step_reuse_inherits():
    rng = np.random.default_rng(14)
    T = 3000
    Ki = rng.standard_normal((T, 128))
    Km = rng.standard_normal((T, 512))
    layers = list(range(20, 40))
    modes = O.layer_modes()
    q_idx = {lay: rng.standard_normal((16, 128)) for lay in layers}
    w_idx = {lay: rng.random(16) for lay in layers}
    q_attn = {lay: rng.standard_normal((64, 512)) * 0.04 for lay in layers}
    swa = {lay: rng.standard_normal((128, 512)) for lay in layers}
    res = O.decode_step(layers, modes, Ki, Km, q_idx, w_idx, q_attn, swa, T, 0, 1.0)
    producer = None
    for lay in layers:
        if modes[lay] in ("Full", "Reindex"):
            producer = lay
        else:
            assert np.array_equal(res[lay][0], res[producer][0])
    assert not np.array_equal(res[20][0], res[24][0])


# ------------------------------------------------------------------ RoPE on the compressed latent
def _rot2(angle):
    """2-D rotation by `angle` radians, from scipy's rotation about the z axis."""
    from scipy.spatial.transform import Rotation
    return Rotation.from_rotvec([0.0, 0.0, angle]).as_matrix()[:2, :2]


def test_rope_preserves_norm_and_leaves_nope_dims():
    """[ARCH] §7: RoPE preserves the norm; only the last 64 of the 512 dims turn, and position 0
    is the identity."""
    rng = np.random.default_rng(71)
    x = rng.standard_normal((6, 512))
    pos = np.array([0, 1, 7, 400, 65535, 1048575])
    y = O.rope_rotate(x, pos)
    assert np.allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)
    pairs = lambda v: v[:, 448:].reshape(len(v), 32, 2)  # noqa: E731
    assert np.allclose(np.linalg.norm(pairs(y), axis=2), np.linalg.norm(pairs(x), axis=2), rtol=1e-13)
    assert np.array_equal(y[:, :448], x[:, :448])
    assert np.array_equal(y[0], x[0])


def test_rope_pairs_turn_like_library_rotations():
    """Pair k of dims (448 + 2k, 449 + 2k) turns counter-clockwise by pos * 160000^(-k/32): pair
    0 by pos radians, pair 16 by pos / 400 (160000^(-1/2) = 1/400), against scipy's rotations."""
    rng = np.random.default_rng(72)
    x = rng.standard_normal((1, 512))
    for pos, k, angle in ((3, 0, 3.0), (400, 16, 1.0), (1000, 16, 2.5), (123457, 0, 123457.0)):
        y = O.rope_rotate(x, [pos])
        want = _rot2(angle) @ x[0, 448 + 2 * k:450 + 2 * k]
        assert np.allclose(y[0, 448 + 2 * k:450 + 2 * k], want, atol=1e-9), (pos, k)
    # the 32 frequencies fall geometrically from 1 by the ratio 160000^(-1/32) per pair
    e = np.zeros((1, 512))
    e[0, 448::2] = 1.0
    ang = np.arctan2(O.rope_rotate(e, [1])[0, 449::2], O.rope_rotate(e, [1])[0, 448::2])
    assert np.allclose(ang[1:] / ang[:-1], 160000.0 ** (-1.0 / 32), rtol=1e-12) and abs(ang[0] - 1.0) < 1e-15


def test_rope_depends_on_relative_position_only():
    """The defining property: the dot product of two rotated rows depends on the position
    difference only, and rotations compose additively."""
    rng = np.random.default_rng(73)
    x, y = rng.standard_normal((2, 1, 512))
    for p, q, s in ((5, 17, 1000), (70000, 3, 12345), (0, 1048575, 7)):
        a = O.rope_rotate(x, [p])[0] @ O.rope_rotate(y, [q])[0]
        b = O.rope_rotate(x, [p + s])[0] @ O.rope_rotate(y, [q + s])[0]
        assert abs(a - b) <= 1e-9 * np.linalg.norm(x) * np.linalg.norm(y)
        assert np.allclose(O.rope_rotate(O.rope_rotate(x, [p]), [q]), O.rope_rotate(x, [p + q]), atol=1e-9)


def test_writer_rope_touches_main_kv_tail_only():
    """With RoPE, the indexer K is the no-RoPE projection and main-KV groups 0..27 (dims < 448)
    keep their codes; the rotated groups differ somewhere."""
    rng = np.random.default_rng(74)
    wkv = rng.standard_normal((64, 512)).astype(np.float32)
    W = (rng.standard_normal((512, 128)) / np.sqrt(512)).astype(np.float32)
    a = O.cache_write_compress(wkv, None, W, 1)
    b = O.cache_write_compress(wkv, None, W, 1, rope_pos=np.arange(1000, 1064))
    assert np.array_equal(a[2], b[2]) and np.array_equal(a[3], b[3])
    assert np.array_equal(a[0][:, :224], b[0][:, :224]) and np.array_equal(a[1][:, :28], b[1][:, :28])
    assert not np.array_equal(a[0][:, 224:], b[0][:, 224:])


# ------------------------------------------------------------------ pool with the window tail
def test_pool_tail_keeps_the_window():
    """[ARCH] §3.3 旁路与边界: with the window tail every one of the newest 128 positions is in
    the pool whatever its block scored; the plain pool is a subset; at most 128 positions are
    added; runs stay 8-aligned and ascending; with every block selected nothing changes."""
    rng = np.random.default_rng(81)
    for vis in (5, 130, 16383, 16385, 16391, 40000, 100001):
        s = rng.standard_normal(vis)
        s[max(0, vis - 200):] -= 100.0           # the newest positions score worst
        m = O.block_maxima(s, vis)
        blk = O.topk_ascending(m, len(m), 2048)
        plain, tail = O.expand_pool(blk, vis), O.expand_pool(blk, vis, tail=True)
        assert len(tail) == 16384 + 160
        ps, ts = set(plain[plain >= 0].tolist()), set(tail[tail >= 0].tolist())
        window = set(range(max(0, vis - 128), vis))
        assert window <= ts and ps <= ts and ts == ps | window
        runs = tail.reshape(-1, 8)
        live = runs[(runs >= 0).any(axis=1)]
        first = np.array([r[r >= 0][0] // 8 for r in live])
        assert np.all(np.diff(first) > 0)
        assert all(((r < 0) | (r // 8 == b)).all() for r, b in zip(live, first))
        if -(-vis // 8) <= 2048:
            assert np.array_equal(tail[:16384], plain) and (tail[16384:] == -1).all()
        elif vis > 20000:
            assert not window <= ps                # the low-scoring window needed the tail
