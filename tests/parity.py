"""Shared helpers of the parity tests: oracle-side inputs and comparisons.

Inputs come from the seeded generator module. The FP4 caches that both sides read are
produced by the oracle's own writer, so no oracle input ever comes from the CUDA path.
Tolerances:
- indices match exactly, except positions whose oracle score lies within TOPK_REL (1e-4,
  relative) of the k-th threshold (the required band);
- attention: max|o - o_ref| / max|o_ref| <= ATTN_REL (2e-3, the required bound);
- cache write: codes equal, except elements within WRITE_REL of a rounding midpoint or a
  scale boundary. The fp32 pipeline (expf, a correctly rounded sqrt and division, 512-term
  fp32 sums) stays within about 1e-6 of the fp64 values, so 1e-5 leaves a 10x margin. The
  excluded fraction itself is bounded (5e-4 of main-KV, 2e-3 of indexer-K elements).
"""
from __future__ import annotations

import numpy as np

import oracle as O
from hierarchical_sparse_attention_index_gb300 import synth

TOPK_REL = 1e-4
ATTN_REL = 2e-3
WRITE_REL = 1e-5
E2M1_MIDS = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])


def f32(bits):
    return synth.bf16_bits_to_f32(bits)


def oracle_cache(seed, layer, batch, T, cap, planted=0, q_plant=None, w_plant=None, scale_fmt=O.SCALE_E8M0):
    """Per-request m=1 cache written by the oracle from seeded N(0,1) latents.

    Returns packed arrays [B][cap][...] (zero padded past T), the dequantised keys per request
    and the planted positions."""
    W = synth.w_idx_bf16(seed, layer)
    kv_q = np.zeros((batch, cap, 256), np.uint8)
    kv_s = np.zeros((batch, cap, 32), np.uint8)
    ik_q = np.zeros((batch, cap, 64), np.uint8)
    ik_s = np.zeros((batch, cap, 4), np.uint8)
    planted_pos = []
    for b in range(batch):
        lat = synth.latents_bf16(seed, layer, b, T)
        if planted:
            planted_pos.append(synth.plant_clusters(lat, W, q_plant[b], w_plant[b], planted, seed, b))
        a, s_, c, d, _, _ = O.cache_write_compress(f32(lat), None, f32(W), 1, scale_fmt)
        kv_q[b, :T], kv_s[b, :T], ik_q[b, :T], ik_s[b, :T] = a, s_, c, d
    return dict(kv_q=kv_q, kv_s=kv_s, ik_q=ik_q, ik_s=ik_s, W=W, planted=planted_pos)


def dequant_index(cache, b, n):
    return O.index_k_dequant(cache["ik_q"][b, :n], cache["ik_s"][b, :n])


def dequant_main(cache, b, n, scale_fmt=O.SCALE_E8M0):
    return O.main_kv_dequant(cache["kv_q"][b, :n], cache["kv_s"][b, :n], scale_fmt)


def check_set_band(gpu_sel, oracle_sel, score, name):
    """Sets may differ only at elements whose oracle score is within TOPK_REL of the threshold."""
    g = set(int(x) for x in gpu_sel)
    o = set(int(x) for x in oracle_sel)
    if g == o:
        return 0
    key = score.astype(np.float32).astype(np.float64)
    tau = min(key[list(o)])
    bad = [x for x in g ^ o if abs(score[x] - tau) > TOPK_REL * abs(tau)]
    assert not bad, f"{name}: {len(g ^ o)} differing, {len(bad)} outside the band (tau={tau}): {bad[:8]}"
    return len(g ^ o)


def check_topk(gpu_row, s, vis, k=512, name="topk"):
    """gpu_row: the kernel's [k] output; s: oracle fp64 scores over positions (>= vis: -inf)."""
    kk = min(k, vis)
    g = gpu_row[gpu_row >= 0]
    assert len(g) == kk, f"{name}: {len(g)} indices, expected {kk}"
    if kk <= 0:                                    # an empty request: every slot is -1
        assert np.all(gpu_row == -1), f"{name}: empty request not -1 filled"
        return 0
    assert np.all(gpu_row[kk:] == -1) and np.all(np.diff(g) > 0), f"{name}: not ascending/-1 padded"
    assert g.min() >= 0 and g.max() < vis
    o = O.topk_ascending(s, vis, k)
    return check_set_band(g, o, s, name)


def check_pool(gpu_pool, s, vis, name="pool"):
    """Structure of the pool plus block-set parity under the band on block maxima."""
    m = O.block_maxima(s, vis)
    nblk = len(m)
    nsel = min(2048, nblk)
    runs = gpu_pool[:8 * nsel].reshape(nsel, 8)
    blocks = runs[:, 0] // 8
    assert np.all(runs[:, 0] >= 0), f"{name}: empty run"
    assert np.all(np.diff(blocks) > 0), f"{name}: blocks not ascending"
    expect = blocks[:, None] * 8 + np.arange(8)[None, :]
    expect = np.where(expect < vis, expect, -1)
    assert np.array_equal(runs, expect), f"{name}: run contents"
    assert np.all(gpu_pool[8 * nsel:] == -1)
    o = O.topk_ascending(m, nblk, 2048)
    return check_set_band(blocks, o, m, name)


def check_pool_tail(gpu_pool, s, vis, name="pool tail"):
    """A pool with the window tail: ascending 8-slot runs; every window block (positions
    [vis - 128, vis)) present, whole or keeping only its window positions; every other run a whole
    selected block; the non-window selected blocks agree with the oracle's block top-2048 within
    the band, and so do window blocks whose run shows whether they were selected."""
    m = O.block_maxima(s, vis)
    nblk = len(m)
    wlo = max(0, vis - 128)
    wb = set(range(wlo // 8, nblk))
    runs = gpu_pool.reshape(-1, 8)
    live = (runs >= 0).any(axis=1)
    nl = int(live.sum())
    assert live[:nl].all() and not live[nl:].any(), f"{name}: runs not contiguous"
    blocks = np.array([r[r >= 0][0] // 8 for r in runs[:nl]], np.int64)
    assert np.all(np.diff(blocks) > 0), f"{name}: blocks not ascending"
    assert wb <= set(blocks.tolist()), f"{name}: window blocks missing"
    picked, known = [], []
    for r, b in zip(runs[:nl], blocks):
        p = 8 * b + np.arange(8)
        whole = np.where(p < vis, p, -1)
        part = np.where((p < vis) & (p >= wlo), p, -1)
        if b in wb:
            assert np.array_equal(r, whole) or np.array_equal(r, part), f"{name}: window run {b}"
            if not np.array_equal(whole, part):
                known.append(int(b))
                if np.array_equal(r, whole):
                    picked.append(int(b))
        else:
            assert np.array_equal(r, whole), f"{name}: run {b}"
            picked.append(int(b))
    o = O.topk_ascending(m, nblk, 2048)
    o_vis = [int(b) for b in o if b not in wb or b in known]
    return check_set_band(np.array(picked), np.array(o_vis), m, name)


def check_attention(o_gpu, o_ref, name="attn"):
    denom = np.max(np.abs(o_ref))
    err = np.max(np.abs(o_gpu.astype(np.float64) - o_ref)) / (denom if denom > 0 else 1.0)
    assert err <= ATTN_REL, f"{name}: rel err {err:.3e} > {ATTN_REL}"
    return err


def _near_mid(v, tol):
    a = np.abs(v)
    return np.any(np.abs(a[..., None] - E2M1_MIDS) <= tol * np.maximum(1.0, a[..., None]), axis=-1)


def unpack_codes(packed):
    packed = np.asarray(packed, np.uint8)
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), np.uint8)
    out[..., 0::2] = packed & 0xF
    out[..., 1::2] = packed >> 4
    return out


def write_exclusions(x64, group, scale_fmt, err_abs):
    """Mask of elements [N, D] whose code the oracle cannot fix to within err_abs of the value:
    near a rounding midpoint of x/s, or in a group whose scale choice is near a boundary."""
    N, D = x64.shape
    g = x64.reshape(N, D // group, group)
    amax = np.abs(g).max(axis=2)
    err = np.broadcast_to(err_abs, x64.shape).reshape(N, D // group, group)
    gerr = err.max(axis=2)
    if scale_fmt == O.SCALE_E8M0:
        cand = 6.0 * O.e8m0_decode(np.arange(255))
    else:
        cand = 6.0 * O.e4m3_decode(np.arange(1, 127))
    near_b = np.min(np.abs(amax[..., None] - cand[None, None, :]), axis=-1) <= gerr
    sb = O.e8m0_scale_byte(amax) if scale_fmt == O.SCALE_E8M0 else O.e4m3_scale_byte(amax)
    s = O.e8m0_decode(sb) if scale_fmt == O.SCALE_E8M0 else O.e4m3_decode(sb)
    v = g / s[..., None]
    near_m = _near_mid(v, 0.0) | (np.min(np.abs(np.abs(v)[..., None] - E2M1_MIDS), axis=-1) <= err / s[..., None])
    mask = near_m | near_b[..., None]
    return mask.reshape(N, D)


def check_write(oc_lat, oc_bytes, gpu, entries, fmt, name):
    """oc_lat: oracle fp64 latents [n,512]; oc_bytes: oracle (kv_q, kv_s, ik_q, ik_s); gpu: same from device."""
    lat, K, W = oc_lat
    n = lat.shape[0]
    # main KV
    ex = write_exclusions(lat, 16, fmt, WRITE_REL * np.maximum(1.0, np.abs(lat)))
    gc = unpack_codes(gpu[0][entries])
    oc = unpack_codes(oc_bytes[0])
    grp_ex = ex.reshape(n, 32, 16).any(axis=2)
    bad = (gc != oc) & ~ex
    assert not bad.any(), f"{name}: {bad.sum()} main-KV codes differ outside the band"
    bad_s = (gpu[1][entries] != oc_bytes[1]) & ~grp_ex
    assert not bad_s.any(), f"{name}: {bad_s.sum()} main-KV scales differ"
    # the band is derived from the fp32 pipeline's error; on the seeded workloads it covers about
    # 1e-4 of the main-KV elements and 4e-4 of the indexer-K elements
    assert ex.mean() < 5e-4, f"{name}: the band excludes {ex.mean():.2e} of the main-KV elements"
    # indexer K (compare element codes in natural order)
    kerr = 4e-6 * (np.abs(lat) @ np.abs(W)) + WRITE_REL * np.abs(K)
    exk = write_exclusions(K, 32, O.SCALE_E8M0, kerr)
    gk = unpack_codes(O.index_k_to_natural(gpu[2][entries]))
    ok_ = unpack_codes(O.index_k_to_natural(oc_bytes[2]))
    bad = (gk != ok_) & ~exk
    assert not bad.any(), f"{name}: {bad.sum()} indexer-K codes differ outside the band"
    bad_s = (gpu[3][entries] != oc_bytes[3]) & ~exk.reshape(n, 4, 32).any(axis=2)
    assert not bad_s.any(), f"{name}: {bad_s.sum()} indexer-K scales differ"
    assert exk.mean() < 2e-3, f"{name}: the band excludes {exk.mean():.2e} of the indexer-K elements"
    return float(ex.mean()), float(exk.mean())


# ------------------------------------------------------------------ oracle writer in a process pool
def write_chunk(args):
    """Pool worker: the oracle's cache writer on one run of tokens. Entries depend only on their
    own tokens (m = 1) or token pair (m = 2), so runs of tokens are independent."""
    wkv, wg, W, m, fmt, keep = args
    kv_q, kv_s, ik_q, ik_s, lat, K = O.cache_write_compress(f32(wkv), None if wg is None else f32(wg), f32(W), m,
                                                            fmt)
    return (kv_q, kv_s, ik_q, ik_s) + ((lat, K) if keep else ())


def oracle_write(pool, wkv, wg, W, m=1, fmt=O.SCALE_E8M0, keep=False, chunk=16384):
    """The oracle's writer over n tokens, split into runs of `chunk` tokens (even, so that m = 2
    pairs stay whole) across a spawn process pool. Returns kv_q, kv_s, ik_q, ik_s (and the fp64
    latent and indexer K with keep=True)."""
    n = wkv.shape[0]
    jobs = [(wkv[i:i + chunk], None if wg is None else wg[i:i + chunk], W, m, fmt, keep) for i in range(0, n, chunk)]
    parts = pool.map(write_chunk, jobs)
    return tuple(np.concatenate([p[k] for p in parts], axis=0) for k in range(len(parts[0])))


class MainRows:
    """Main-KV rows of one request, dequantised on demand (K_main[sel] for a list of positions),
    so that attention references at 1M positions never dequantise the whole request."""

    def __init__(self, kv_q, kv_s, fmt=O.SCALE_E8M0):
        self.kv_q, self.kv_s, self.fmt = kv_q, kv_s, fmt

    def __getitem__(self, sel):
        sel = np.asarray(sel, np.int64)
        return O.main_kv_dequant(self.kv_q[sel], self.kv_s[sel], self.fmt)
