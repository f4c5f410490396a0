"""Plain fp64 CPU oracle for the CSA2 hierarchical sparse indexer, sparse attention and
compressed-cache write (DeepSeek-V4.1-Flash decode hot path).

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import or run this module. The product path
never does. It shares no code, table or constant with the CUDA path; its inputs are plain
numpy arrays.

Everything is the plain definition: numpy fp64, with a library matmul or sort used as a
single step and no blocking, fusion or reordering. Where a floating-point value decides an
integer (an FP4 code, a scale exponent, a top-k membership), the decision is taken on the
value rounded to float32. That is the precision the pages give for the compressor ("m > 1
runs in fp32"), and the kernel's precision for the scores.

Sources. The pages are cited by tag, title and section:

- [890B]  jokeuncle.pages.dev, "两张架构图里藏着 890 字节：把 DeepSeek V4.1 Flash 的 43 层排班表算出来"
- [COST]  weigao.cc, "DeepSeek V4.1 Flash：从架构到推理成本"
- [CED]   syt-nju.github.io, "DeepSeek-V4.1-Flash：为什么读输入只激活 8B，写输出要 16B"
- [ARCH]  ggaaooppeenngg.github.io, "DeepSeek-V4.1-Flash 架构解析：KV Cache 压缩的极限在哪里"
- [10100] 10100.com, DeepSeek-V4.1-Flash 背景 / Architecture / 层次化稀疏索引器

Parity status of each part:

- pinned: the format decoders, quantiser, byte counts, layer schedule, score, top-k,
  block/pool, reindex, attention and cache write (see tests/test_oracle_pins.py);
- parity unpinned (choices the pages leave open, documented as such): the E8M0/E4M3 scale
  rule, the nibble order, the SWA row mapping and the tie order. The tests fix these as
  conventions, not as facts.
"""
from __future__ import annotations

import math

import numpy as np

# ---------------------------------------------------------------------------------------
# Constants of the configuration ([890B] §二 table of config.json keys; [ARCH] §3.3)
# ---------------------------------------------------------------------------------------
D_LATENT = 512          # head_dim of the compressed main KV            [890B] §三 事实一
D_INDEX = 128           # index_head_dim                                [890B] §三 事实二
H_INDEX = 16            # indexer heads (lineage: DeepSeek-V3.2 indexer; workload definition)
H_ATTN = 64             # query heads x 512                             [ARCH] §1 table
MAIN_GROUP = 16         # channels per main-KV scale                    [890B] §三 事实一
INDEX_GROUP = 32        # channels per indexer-K scale                  [890B] §三 事实二
INDEX_TOPK = 512        # index_topk                                    [890B] 注意力实际有多稀
CAND_BLOCKS = 2048      # candidate_topk_blocks                         [890B] §二 table
CAND_BLOCK = 8          # candidate_block_size                          [890B] 候选池让深层索引器…
POOL_SLOTS = CAND_BLOCKS * CAND_BLOCK   # 16,384                        [CED] Figure 5
SWA_W = 128             # sliding_window                                [890B] §二 table
POOL_TAIL_SLOTS = 160   # pool slots past POOL_SLOTS with the window tail: the <= 17 window blocks, as 5 x 32
RMS_EPS = 1e-6
ROPE_THETA = 160000.0   # RoPE base of the compressed latent           [ARCH] §3.2 压缩 RoPE
ROPE_DIMS = 64          # rotary dims: the last 64 of 512 (the 448 B NoPE + 128 B RoPE page layout) [ARCH] §7

SCALE_E8M0 = 0
SCALE_E4M3 = 1


# ---------------------------------------------------------------------------------------
# Number formats. E2M1 value + scale per group: [890B] §三; [CED] "FP4 主 KV 缓存"; [ARCH] §7
# ---------------------------------------------------------------------------------------
def e2m1_decode(nibble) -> np.ndarray:
    """FP4 E2M1: 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit, no inf/NaN.
    e = 0 is subnormal (m * 0.5); e > 0 gives (1 + m/2) * 2^(e-1)."""
    n = np.asarray(nibble, dtype=np.int64) & 0xF
    s = (n >> 3) & 1
    e = (n >> 1) & 3
    m = n & 1
    mag = np.where(e == 0, m * 0.5, (1.0 + m * 0.5) * np.exp2(e - 1.0))
    return np.where(s == 1, -mag, mag).astype(np.float64)


def e8m0_decode(byte) -> np.ndarray:
    """E8M0 scale: 2^(b - 127); b = 255 is NaN."""
    b = np.asarray(byte, dtype=np.int64)
    v = np.exp2(b.astype(np.float64) - 127.0)
    return np.where(b == 255, np.nan, v)


def e4m3_decode(byte) -> np.ndarray:
    """FP8 E4M3 (the 'fn' variant): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits;
    e = 0 is subnormal (m/8 * 2^-6); exponent 15 with mantissa 7 is NaN; no infinities."""
    b = np.asarray(byte, dtype=np.int64) & 0xFF
    s = (b >> 7) & 1
    e = (b >> 3) & 0xF
    m = b & 7
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag)


# Magnitude intervals of round-to-nearest-even onto the E2M1 grid {0,.5,1,1.5,2,3,4,6}.
# A value on a midpoint goes to the neighbour whose mantissa bit is 0 ("even"), and
# anything above 6 saturates to 6.
#   [0, .25] -> 0   (.25, .75) -> .5   [.75, 1.25] -> 1   (1.25, 1.75) -> 1.5
#   [1.75, 2.5] -> 2   (2.5, 3.5) -> 3   [3.5, 5] -> 4   (5, inf) -> 6
def e2m1_encode(v) -> np.ndarray:
    """float32 value -> E2M1 nibble, round to nearest even, saturating, -0 stored as +0."""
    v = np.asarray(v, dtype=np.float32)
    a = np.abs(v).astype(np.float64)
    code = np.zeros(a.shape, dtype=np.int64)
    code = np.where(a > 0.25, 1, code)
    code = np.where(a >= 0.75, 2, code)
    code = np.where(a > 1.25, 3, code)
    code = np.where(a >= 1.75, 4, code)
    code = np.where(a > 2.5, 5, code)
    code = np.where(a >= 3.5, 6, code)
    code = np.where(a > 5.0, 7, code)
    sign = np.where((v < 0) & (code != 0), 8, 0)
    return (code | sign).astype(np.uint8)


def _e4m3_positive_table() -> np.ndarray:
    vals = e4m3_decode(np.arange(1, 127))          # 0x01..0x7E: every finite positive value
    return vals


def e8m0_scale_byte(amax) -> np.ndarray:
    """Scale rule (a reading; the pages give none): the smallest power of two s = 2^e with
    6*s >= amax, so x/s never leaves the E2M1 range; amax = 0 gives byte 0 (2^-127).
    The comparison is exact."""
    amax = np.asarray(amax, dtype=np.float64)
    with np.errstate(divide="ignore"):
        e = np.ceil(np.log2(np.where(amax > 0, amax, 1.0) / 6.0))
    e = np.clip(e, -127, 127)
    for _ in range(2):       # exact correction of the log2 estimate
        e = np.where((e > -127) & (6.0 * np.exp2(e - 1) >= amax), e - 1, e)
        e = np.where((e < 127) & (6.0 * np.exp2(e) < amax), e + 1, e)
    e = np.where(amax > 0, e, -127)
    return (e + 127).astype(np.uint8)


def e4m3_scale_byte(amax) -> np.ndarray:
    """E4M3 variant of the scale rule: the smallest positive E4M3 value s with 6*s >= amax
    (amax/6 rounded up onto the E4M3 grid). It saturates at 448; amax = 0 gives the
    smallest subnormal."""
    amax = np.asarray(amax, dtype=np.float64)
    tab = _e4m3_positive_table()
    idx = np.searchsorted(6.0 * tab, amax, side="left")
    idx = np.minimum(idx, len(tab) - 1)
    return (idx + 1).astype(np.uint8)


def quantise_groups(x32: np.ndarray, group: int, scale_fmt: int):
    """Group FP4 quantisation of float32 rows [N, D] -> (packed codes [N, D/2], scales [N, D/group]).

    Per group: amax -> scale byte -> code = RNE_E2M1(x / s), the division taken in float32.
    No second-level global scale ([CED] "FP4 主 KV 缓存": 类似 NVFP4，但去掉了第二级全局缩放).
    Packing (a layout choice): byte j holds element 2j in its low nibble and 2j+1 in its high nibble."""
    x32 = np.asarray(x32, dtype=np.float32)
    N, D = x32.shape
    g = x32.reshape(N, D // group, group)
    amax = np.abs(g).max(axis=2).astype(np.float64)
    if scale_fmt == SCALE_E8M0:
        sb = e8m0_scale_byte(amax)
        s = e8m0_decode(sb)
    else:
        sb = e4m3_scale_byte(amax)
        s = e4m3_decode(sb)
    v = g / s.astype(np.float32)[:, :, None]       # float32 / float32, IEEE rounded
    codes = e2m1_encode(v).reshape(N, D)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return packed, sb.astype(np.uint8)


def dequant_groups(packed: np.ndarray, scales: np.ndarray, group: int, scale_fmt: int) -> np.ndarray:
    """Inverse of the packing: value = E2M1(code) * scale, in fp64 ([ARCH] §7: 注意力前反量化)."""
    packed = np.asarray(packed, dtype=np.uint8)
    N = packed.shape[0]
    codes = np.empty((N, packed.shape[1] * 2), dtype=np.uint8)
    codes[:, 0::2] = packed & 0xF
    codes[:, 1::2] = packed >> 4
    vals = e2m1_decode(codes)
    s = e8m0_decode(scales) if scale_fmt == SCALE_E8M0 else e4m3_decode(scales)
    return (vals.reshape(N, -1, group) * s[:, :, None]).reshape(N, -1)


def main_kv_dequant(kv_q, kv_s, scale_fmt=SCALE_E8M0):
    """Main-KV entry: 512 x E2M1 + one scale byte per 16 channels = 288 B ([890B] §三 事实一)."""
    return dequant_groups(kv_q, kv_s, MAIN_GROUP, scale_fmt)


# Indexer-K byte order (a layout choice; the pages fix the value format only). The stored
# byte 16t + 2s + i holds the logical byte 8s + 2t + i, whose low nibble is element
# 2(8s + 2t + i) and high nibble the next element.
def _fragment_perm():
    perm = np.empty(64, np.int64)          # perm[stored] = logical
    for t in range(4):
        for s in range(8):
            for i in range(2):
                perm[16 * t + 2 * s + i] = 8 * s + 2 * t + i
    return perm


def index_k_to_stored(packed_natural):
    """Natural packing (byte j = elements 2j, 2j+1) -> stored fragment order."""
    packed_natural = np.asarray(packed_natural, np.uint8)
    return packed_natural[:, _fragment_perm()]


def index_k_to_natural(stored):
    """Stored fragment order -> natural packing."""
    stored = np.asarray(stored, np.uint8)
    out = np.empty_like(stored)
    out[:, _fragment_perm()] = stored
    return out


def index_k_dequant(ik_q, ik_s):
    """Indexer-K entry: 128 x E2M1 in fragment order + one E8M0 per 32 channels = 68 B
    ([890B] §三 事实二)."""
    return dequant_groups(index_k_to_natural(ik_q), ik_s, INDEX_GROUP, SCALE_E8M0)


def swa_decode(rows_u8):
    """SWA tail rows are FP8 E4M3 with no scale ([CED] "FP4 主 KV 缓存": SWA KV 仍保留 FP8; [ARCH] §4.1)."""
    return e4m3_decode(rows_u8)


# ---------------------------------------------------------------------------------------
# Byte accounting ([890B] §三; [COST] §4)
# ---------------------------------------------------------------------------------------
def entry_bytes():
    """(main-KV bytes, indexer-K bytes) of one compressed slot, counted from the packer."""
    kv_q, kv_s = quantise_groups(np.zeros((1, D_LATENT), np.float32), MAIN_GROUP, SCALE_E8M0)
    ik_q, ik_s = quantise_groups(np.zeros((1, D_INDEX), np.float32), INDEX_GROUP, SCALE_E8M0)
    return kv_q.nbytes + kv_s.nbytes, ik_q.nbytes + ik_s.nbytes


def global_kv_bytes_per_token(ratios_of_kv_sources, k_owner_layers=None):
    """Sum over cache-owning layers of (bytes per slot) / (compress ratio).

    Only KV-source layers own an indexer-K buffer ([890B] §三 "owns_k"). Passing extra
    layers in ``k_owner_layers`` models the wrong count that also stores K for Reindex
    layers."""
    main, idx = entry_bytes()
    total = sum((main + idx) / r for r in ratios_of_kv_sources)
    if k_owner_layers:
        total += idx * len(k_owner_layers)
    return total


# ---------------------------------------------------------------------------------------
# Layer schedule ([890B] §二 43-layer table; [COST] §3.1; [ARCH] §3.2; [CED] Figure 3)
# ---------------------------------------------------------------------------------------
KV_SOURCE_LAYERS = (2, 8, 14, 20)
INDEX_SOURCE_LAYERS = (2, 8, 14, 20, 24, 28, 32, 36)
N_BACKBONE = 40
N_DRAFT = 3


def compress_ratios():
    """43 entries: layers 0-1 and the three draft layers are SWA-only (0), the encoder
    2-19 uses 2, the decoder 20-39 uses 1 ([890B] §二 table)."""
    return [0, 0] + [2] * 18 + [1] * 20 + [0] * N_DRAFT


def layer_modes():
    """Mode of every layer: 'SWA', 'Full', 'Reindex' or 'Reuse'.

    Full = KV source (stores KV and K, scores everything); Reindex = index source that is
    not a KV source (rescoring the pool); Reuse = every other compressed layer
    ([CED] Figure 4; [ARCH] §3.2 table)."""
    modes = []
    for layer, r in enumerate(compress_ratios()):
        if r == 0:
            modes.append("SWA")
        elif layer in KV_SOURCE_LAYERS:
            modes.append("Full")
        elif layer in INDEX_SOURCE_LAYERS:
            modes.append("Reindex")
        else:
            modes.append("Reuse")
    return modes


def decoder_step_counts(first=20, last=39):
    """(full scores, pool rescores, inherits) per decode step over the decoder layers
    ([ARCH] §3.3: 1 次全量打分 + 4 次池内打分 + 15 次继承)."""
    m = layer_modes()[first:last + 1]
    return m.count("Full"), m.count("Reindex"), m.count("Reuse")


# ---------------------------------------------------------------------------------------
# Indexer scoring ([CED] Figure 5; [ARCH] §3.3; [10100] 层次化稀疏索引器)
# ---------------------------------------------------------------------------------------
def index_scores(q, w, K, vis):
    """s[t] = sum_h w_h * ReLU(q_h . k_t) for t < vis; -inf beyond.

    q: [16, 128] (the bf16 values), w: [16], K: [T, 128] dequantised keys, vis: int.
    The per-head weighted ReLU sum follows the DeepSeek-V3.2 indexer lineage that the
    pages name; the formula itself is the workload's definition."""
    q = np.asarray(q, np.float64)
    w = np.asarray(w, np.float64)
    K = np.asarray(K, np.float64)
    T = K.shape[0]
    dots = K[:min(vis, T)] @ q.T                          # [vis, 16]
    s = np.full(T, -np.inf)
    s[:min(vis, T)] = np.maximum(dots, 0.0) @ w
    return s


def _rank_key(s):
    """The float32 value on which a membership decision is taken."""
    return np.asarray(s, np.float64).astype(np.float32).astype(np.float64)


def topk_ascending(s, n_valid, k):
    """Indices of the min(k, n_valid) largest entries of s[:n_valid], ordered by
    (float32(s) descending, index ascending) and returned in ascending index order."""
    n_valid = int(n_valid)
    kk = min(k, n_valid)
    if kk <= 0:
        return np.zeros(0, np.int64)
    key = _rank_key(s[:n_valid])
    order = np.lexsort((np.arange(n_valid), -key))       # primary: key desc, then index asc
    return np.sort(order[:kk])


def block_maxima(s, vis):
    """m_b = max over the visible positions of block b = [8b, 8b+8) ([ARCH] §3.3: 每块取块内最大索引分).
    Blocks align to position 0; a partial last block uses its visible positions."""
    vis = int(vis)
    nblk = -(-vis // CAND_BLOCK)
    m = np.full(nblk, -np.inf)
    for b in range(nblk):
        m[b] = np.max(s[b * CAND_BLOCK:min(vis, (b + 1) * CAND_BLOCK)])
    return m


def expand_pool(blocks, vis, tail=False):
    """Candidate pool: each selected block (ascending) contributes 8 slots 8b..8b+7, with
    positions >= vis written as -1. Slots beyond the selected blocks are -1. The size is
    min(2048, ceil(vis/8))*8 live slots out of 16,384 ([CED] Figure 5; [ARCH] §3.3).

    With tail ([ARCH] §3.3 旁路与边界: the newest tokens of the sliding window skip the funnel
    and are merged at the tail of the expanded pool, so they are not lost while their block is
    still filling): the blocks holding positions [vis - 128, vis) join the selected ones, and a
    window block the selection did not pick contributes only its positions >= vis - 128. The
    union stays in ascending block order (the window blocks are the last ones, at the tail), in
    POOL_SLOTS + POOL_TAIL_SLOTS slots. That the window joins by whole 8-slot runs, deduplicated
    against the selected blocks, is a reading."""
    vis = int(vis)
    sel = set(int(b) for b in blocks)
    wlo = max(0, vis - SWA_W)
    run_blocks = sel | (set(range(wlo // CAND_BLOCK, -(-vis // CAND_BLOCK))) if tail else set())
    pool = np.full(POOL_SLOTS + (POOL_TAIL_SLOTS if tail else 0), -1, np.int64)
    for i, b in enumerate(sorted(run_blocks)):
        p = b * CAND_BLOCK + np.arange(CAND_BLOCK)
        keep = (p < vis) & ((p >= wlo) | (b in sel))
        pool[i * CAND_BLOCK:(i + 1) * CAND_BLOCK] = np.where(keep, p, -1)
    return pool


def index_full(q, w, K, vis, topk=INDEX_TOPK, n_blocks=CAND_BLOCKS, tail=False):
    """Full layer: one score pass over every visible entry, then two top-k's side by side
    on the same scores: a position top-512 for its own attention and a block top-2048
    (block max) whose blocks expand into the shared candidate pool
    ([ARCH] §3.3 时序澄清; [CED] Figure 5 left/middle).

    Returns (topk positions [512] ascending, -1 padded; pool [16384, or 16544 with the window
    tail]; scores; block maxima)."""
    s = index_scores(q, w, K, vis)
    pos = topk_ascending(s, vis, topk)
    out = np.full(topk, -1, np.int64)
    out[:len(pos)] = pos
    m = block_maxima(s, vis)
    blk = topk_ascending(m, len(m), n_blocks)
    pool = expand_pool(blk, vis, tail)
    return out, pool, s, m


def index_reindex(q, w, K, pool, vis, topk=INDEX_TOPK):
    """Reindex layer: score only the candidate-pool slots with the layer's own indexer Q
    and weights, then take its own top-512 ([CED] Figure 5 right; [ARCH] §3.3 池内过滤).

    Returns (positions [512] ascending, -1 padded; slot scores)."""
    pool = np.asarray(pool, np.int64)
    valid = (pool >= 0) & (pool < vis)
    s_slot = np.full(len(pool), -np.inf)
    if valid.any():
        s_all = index_scores(q, w, K, vis)
        s_slot[valid] = s_all[pool[valid]]
    n_valid = int(valid.sum())
    key = _rank_key(s_slot)
    idx_valid = np.nonzero(valid)[0]
    kk = min(topk, n_valid)
    out = np.full(topk, -1, np.int64)
    if kk > 0:
        kv = key[idx_valid]
        pv = pool[idx_valid]
        order = np.lexsort((pv, -kv))      # key desc, then position asc
        out[:kk] = np.sort(pv[order[:kk]])
    return out, s_slot


# ---------------------------------------------------------------------------------------
# Sparse attention ([CED] Figure 4: Selected Main KV ⊕ SWA KV -> Core Attention;
# [890B] 注意力实际有多稀: 128 + 512 = 640 positions)
# ---------------------------------------------------------------------------------------
def attention_rows(K_main, topk, swa_rows, q_index, vis):
    """The keys query ``q_index`` attends to: the valid top-k main-KV rows, then the SWA tail
    rows [q_index, q_index + W). SWA row q_index + r holds position vis - W + r; rows at
    negative positions are absent (a reading for contexts shorter than the window).
    K = V = the 512-d latent (MLA style)."""
    sel = [int(t) for t in topk if 0 <= t < vis]
    rows = [K_main[sel]] if sel else []
    r = np.arange(SWA_W)
    keep = (vis - SWA_W + r) >= 0
    rows.append(swa_rows[q_index + r[keep]])
    return np.concatenate(rows, axis=0) if rows else np.zeros((0, D_LATENT))


def sparse_attention(q, rows, sm_scale):
    """o_h = sum_j softmax_j(sm_scale * q_h . k_j) * k_j with log-sum-exp stabilisation.
    q: [64, 512] (the bf16 values); rows: [n, 512]. With no rows the output is 0."""
    q = np.asarray(q, np.float64)
    rows = np.asarray(rows, np.float64)
    if rows.shape[0] == 0:
        return np.zeros((q.shape[0], rows.shape[1] if rows.ndim == 2 else D_LATENT))
    logits = sm_scale * (q @ rows.T)                     # [64, n]
    mx = logits.max(axis=1, keepdims=True)
    p = np.exp(logits - mx)
    p /= p.sum(axis=1, keepdims=True)
    return p @ rows


# ---------------------------------------------------------------------------------------
# Compressor and cache write ([890B] §四.1 softmax gating, fp32 for m > 1;
# [ARCH] §3.2 Z 的计算; [CED] "CSA2" 压缩器去掉重叠窗口和绝对位置编码)
# ---------------------------------------------------------------------------------------
def compress_pool(wkv, wgate, m):
    """Per channel, a softmax over the m tokens of a group, then the weighted sum. m = 1 has
    no gating path: the entry is the projection itself ([ARCH] §3.2). Non-overlapping groups
    of m consecutive tokens; a trailing incomplete group is not written."""
    x = np.asarray(wkv, np.float64)
    n = (x.shape[0] // m) * m
    if m == 1:
        return x[:n].copy()
    g = np.asarray(wgate, np.float64)[:n].reshape(-1, m, x.shape[1])
    x = x[:n].reshape(-1, m, x.shape[1])
    g = g - g.max(axis=1, keepdims=True)
    p = np.exp(g)
    p /= p.sum(axis=1, keepdims=True)
    return (x * p).sum(axis=1)


def rms_norm(x, eps=RMS_EPS):
    """RMSNorm with unit gain: x / sqrt(mean(x^2) + eps) ([ARCH] §3.2, §7)."""
    x = np.asarray(x, np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)


def rope_rotate(lat, positions, theta=ROPE_THETA):
    """RoPE on the last ROPE_DIMS dims of each row ([ARCH] §3.2: RMSNorm, the no-RoPE version,
    then compressed RoPE with theta = 160000; [ARCH] §7: RoPE preserves the norm). Pair
    (448 + 2k, 449 + 2k), k = 0..31, turns by positions[row] * theta^(-2k/64) radians:
    (a, b) -> (a cos - b sin, a sin + b cos). The interleaved pairing and the position (the
    entry's index in the request's cache) are readings; the pages give neither."""
    x = np.array(lat, np.float64, copy=True)
    lo = D_LATENT - ROPE_DIMS
    k = np.arange(ROPE_DIMS // 2, dtype=np.float64)
    freq = theta ** (-2.0 * k / ROPE_DIMS)
    ang = np.asarray(positions, np.float64)[:, None] * freq[None, :]
    c, s_ = np.cos(ang), np.sin(ang)
    a = x[:, lo::2].copy()
    b = x[:, lo + 1::2].copy()
    x[:, lo::2] = a * c - b * s_
    x[:, lo + 1::2] = a * s_ + b * c
    return x


def cache_write_compress(wkv, wgate, w_idx, m, scale_fmt=SCALE_E8M0, rope_pos=None):
    """Entries of one request: pooled latent -> RMSNorm -> FP4 main KV (group 16), and
    indexer K = latent . W_idx -> FP4 (group 32, E8M0)
    ([890B] §三; [CED] CSA2 "indexer K 直接由主 KV 投影"; [ARCH] §3.1).

    With rope_pos (the entries' positions) the main KV holds the latent after RoPE and the
    indexer K is still projected from the latent before it ([ARCH] §3.2 names the no-RoPE
    version before the compressed RoPE step; that K comes from it is a reading).
    Returns (kv_q [n,256], kv_s [n,32], ik_q [n,64], ik_s [n,4], main-KV latent fp64, K fp64)."""
    lat = rms_norm(compress_pool(wkv, wgate, m))
    main = lat if rope_pos is None else rope_rotate(lat, rope_pos)
    kv_q, kv_s = quantise_groups(main.astype(np.float32), MAIN_GROUP, scale_fmt)
    K = lat @ np.asarray(w_idx, np.float64)
    ik_nat, ik_s = quantise_groups(K.astype(np.float32), INDEX_GROUP, SCALE_E8M0)
    return kv_q, kv_s, index_k_to_stored(ik_nat), ik_s, main, K


# ---------------------------------------------------------------------------------------
# One decode step over the decoder layers ([ARCH] §3.3; [COST] §3.2; [CED] Figure 4)
# ---------------------------------------------------------------------------------------
def decode_step(layers, modes, K_index, K_main, q_idx, w_idx, q_attn, swa, vis, q_index, sm_scale):
    """Run the schedule for one query of one request.

    Full scores everything and builds the pool; Reindex rescores the pool; Reuse
    inherits the latest indices. Every layer attends with its own Q and SWA tail.
    The per-layer inputs are dicts keyed by layer id. Returns a dict of per-layer
    (topk, output) plus the pool."""
    res = {}
    topk = None
    pool = None
    for layer in layers:
        mode = modes[layer]
        if mode == "Full":
            topk, pool, _, _ = index_full(q_idx[layer], w_idx[layer], K_index, vis)
        elif mode == "Reindex":
            topk, _ = index_reindex(q_idx[layer], w_idx[layer], K_index, pool, vis)
        rows = attention_rows(K_main, topk, swa[layer], q_index, vis)
        res[layer] = (topk.copy(), sparse_attention(q_attn[layer], rows, sm_scale))
    res["pool"] = pool
    return res


def pool_size(vis):
    """Live pool slots: min(2048, ceil(vis/8)) * 8 ([COST] §3.2; [CED] Figure 5)."""
    return min(CAND_BLOCKS, math.ceil(vis / CAND_BLOCK)) * CAND_BLOCK
