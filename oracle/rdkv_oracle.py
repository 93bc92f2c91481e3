"""Plain CPU oracle of the RDKV hot path (weights, allocation, TriZone pack, decode).

TEST INFRASTRUCTURE ONLY: imported by tests/, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py``; never by the library.  It shares no code with
the CUDA sources.

Sources (the pages are summaries; every step they leave open follows the
project's written reading, listed at the end of this header):

* "RDKV - rate-distortion bit allocation for joint KV eviction and
  quantisation" (gist.science/ko/paper/2605.08317):
  section 2.1 (token weight w_t, channel weight w_c, the objective),
  section 2.2 (discrete reverse water-filling over {0,2,4,8,16}; steps 1-3),
  section 2.3 (TriZone layout: zone A packed 2/4/8-bit rows grouped by width,
  zone B fp16 V rows of 16-bit tokens, zone C fp16 rows of new tokens).
* "Matematika KV Cache Compression" (aistudio.id), section "Anatomi Krisis"
  (the KV-size formula 2*L*H_kv*D*P*N) and section "Solusi 3" (asymmetric
  min-max quantiser).

Arithmetic: weights, spreads and attention in float64; breakpoints, gains and
the quantiser in IEEE float32 / float16 exactly as the encoding fixes them, so
that the packed bytes and the bit allocation are reproducible bit for bit.

Parity pins (tests/test_oracle_pins.py): every function below is pinned by a
closed form, an invariant, a library special case or brute force; none is
"parity unpinned".  The end-to-end accuracy of the method on real tasks is not
an oracle function and is out of scope (it needs datasets and trained models).

Readings where the pages are silent (each is a project decision):
 R1 GQA: w_t of KV head j sums over the G query heads of its group.
 R2 The last W prompt tokens (the window) go to zone C in fp16 and are not
    allocated; the allocatable prefix is tokens [0, N-W).
 R3 sigma_u (undefined on the page) = population standard deviation of the
    unit's values: a V row over its D elements; a K channel over the kept
    prefix tokens.  The printed linear form g_u * 2**-b_u is kept.
 R4 One water level per sequence, pooled over KV heads; budget
    B = floor(avg_bits * units); slack left unused.
 R5 At a breakpoint the cheaper width wins (strict >); g = 0 gives 0 bits.
 R6 Quantiser groups: 32 consecutive channels of a V row; for K, one channel
    over every kept prefix token of its (sequence, KV head): the per-channel K
    groups the quantiser statement names.  fp16 scale and zero.
 R7 16-bit K channels are stored raw in fp16 inside zone A; 0-bit K channels
    are dropped and contribute nothing to the logits.
 R8 Byte layout of the zones: see ``pack``.
 R9 Decode: see ``decode`` (scale 1/sqrt(D), every token of zones A, B, C).
 R10 Zone-C re-compression (new tokens joining zones A and B): see the last
    section, above ``attention_lse``.
"""
from __future__ import annotations

import math

import numpy as np

WIDTHS = np.array([0, 2, 4, 8, 16], dtype=np.uint8)
STEP_BITS = np.diff(WIDTHS.astype(np.int64))            # bits gained by each upgrade: 2, 2, 4, 8
V_CLASSES = (2, 4, 8, 16)                                # zone order of kept tokens
K_CLASSES = (16, 8, 4, 2)                                # slot order of kept channels
TILE = 32                                                # tokens per zone-A tile
GROUP = 32                                               # channels per V quantiser group


# ---------------------------------------------------------------------------
# KV-size formula (aistudio.id, "Anatomi Krisis")
# ---------------------------------------------------------------------------
def kv_cache_bytes(n_layers, h_kv, head_dim, bytes_per_elem, n_tokens):
    """Bytes of a full K+V cache: 2 * L * H_kv * D * P * N."""
    return 2 * n_layers * h_kv * head_dim * bytes_per_elem * n_tokens


# ---------------------------------------------------------------------------
# Step 1: distortion weights (RDKV section 2.1; computed once after prefill,
# section 2.2 step 1)
# ---------------------------------------------------------------------------
def _f64(x):
    return np.asarray(x, dtype=np.float64)


def _masked_logits(q_rows, k_all, first_row, head_dim):
    """Causal logits q_tau . k_t / sqrt(D) for rows tau = first_row.., -inf where t > tau."""
    s = q_rows @ k_all.T / math.sqrt(head_dim)
    taus = np.arange(first_row, first_row + q_rows.shape[0])[:, None]
    s[np.arange(k_all.shape[0])[None, :] > taus] = -np.inf
    return s


def token_weights(q, k, first_row=0, row_block=512):
    """V-token weight w_t = sum over query positions tau (and the G heads of the
    group, R1) of the softmax attention a_{tau,t}.

    q [N, H_q, D], k [N, H_kv, D] -> w [H_kv, N] float64.  Only query rows
    tau >= first_row contribute, which is exact for every t >= first_row
    (a_{tau,t} = 0 for tau < t).
    """
    q64, k64 = _f64(q), _f64(k)
    N, Hq, D = q64.shape
    Hkv = k64.shape[1]
    G = Hq // Hkv
    w = np.zeros((Hkv, N))
    for h in range(Hq):
        j = h // G
        for r0 in range(first_row, N, row_block):
            r1 = min(N, r0 + row_block)
            s = _masked_logits(q64[r0:r1, h, :], k64[:, j, :], r0, D)
            a = np.exp(s - s.max(axis=1, keepdims=True))
            a /= a.sum(axis=1, keepdims=True)
            w[j] += a.sum(axis=0)
    return w


def row_lse(q, k, h, rows):
    """log sum_{t <= tau} exp(q_tau,h . k_t / sqrt(D)) for the listed query rows."""
    q64, k64 = _f64(q), _f64(k)
    N, Hq, D = q64.shape
    j = h // (Hq // k64.shape[1])
    out = np.empty(len(rows))
    for i, tau in enumerate(rows):
        s = q64[tau, h, :] @ k64[: tau + 1, j, :].T / math.sqrt(D)
        m = s.max()
        out[i] = m + math.log(np.exp(s - m).sum())
    return out


def channel_weights(q, k):
    """K-channel weight w_c = ||Q_{:,c}|| * ||K_{:,c}|| / sqrt(d) per KV head.

    Q_{:,c} stacks the G query heads of the group over all N positions (R1);
    K_{:,c} runs over all N tokens.  Returns [H_kv, D] float64.
    """
    q64, k64 = _f64(q), _f64(k)
    N, Hq, D = q64.shape
    Hkv = k64.shape[1]
    G = Hq // Hkv
    qn = np.sqrt((q64 ** 2).reshape(N, Hkv, G, D).sum(axis=(0, 2)))
    kn = np.sqrt((k64 ** 2).sum(axis=0))
    return qn * kn / math.sqrt(D)


def value_spread(v):
    """sigma of each V row (R3): population std over its D elements.  [H_kv, N] float64."""
    v64 = _f64(v)                                       # [N, H_kv, D]
    mean = v64.mean(axis=2, keepdims=True)
    return np.sqrt(((v64 - mean) ** 2).mean(axis=2)).T


def token_gains(w_tok, sigma_tok, n_prefix):
    """g_t = fl32(fl32(w_t) * fl32(sigma_t)) on the allocatable prefix."""
    w32 = np.asarray(w_tok[:, :n_prefix], dtype=np.float32)
    s32 = np.asarray(sigma_tok[:, :n_prefix], dtype=np.float32)
    return w32 * s32


def score(q, k, v, window):
    """All step-1 outputs for one sequence, rounded to float32 as the library returns them."""
    N = q.shape[0]
    w_tok = token_weights(q, k)
    sig = value_spread(v)
    return dict(
        w_tok=w_tok.astype(np.float32),
        w_chan=channel_weights(q, k).astype(np.float32),
        sigma_tok=sig.astype(np.float32),
        g_tok=token_gains(w_tok, sig, N - window),
    )


# ---------------------------------------------------------------------------
# Steps 2 and 3: discrete reverse water-filling (RDKV section 2.2)
# ---------------------------------------------------------------------------
# The distortion of a unit at width b is g * 2**-b (section 2.1 objective).
# Moving from width b_k to b_{k+1} removes g * (2**-b_k - 2**-b_{k+1}) of
# distortion for (b_{k+1} - b_k) bits: the slope per bit below, times g.
SLOPES = np.array(
    [(2.0 ** -int(b0) - 2.0 ** -int(b1)) / (int(b1) - int(b0)) for b0, b1 in zip(WIDTHS[:-1], WIDTHS[1:])],
    dtype=np.float32)


def breakpoints(g):
    """beta_{u,k} = fl32(g_u * slope_k): the water levels at which unit u buys upgrade k."""
    g = np.asarray(g, dtype=np.float32).reshape(-1)
    return g[:, None] * SLOPES[None, :]


def widths_at(beta, lam):
    """Lagrangian choice at water level lam: every upgrade whose breakpoint is strictly above lam (R5)."""
    return WIDTHS[(beta > np.float32(lam)).sum(axis=1)]


def budget_bits(avg_bits, n_units):
    """B = floor(avg_bits * units) (R4); avg_bits arrives as float32."""
    return int(math.floor(float(np.float32(avg_bits)) * float(n_units)))


def waterfill(g, avg_bits):
    """Multiple-choice knapsack over {0,2,4,8,16} by Lagrangian relaxation.

    Returns (bits uint8 [U], lambda float32): lambda is the smallest
    non-negative float32 water level whose total width fits the budget
    B = floor(avg_bits * U).  Found exactly: the bit total only changes at
    breakpoints, so the candidates are 0 and the breakpoint values, sorted.
    """
    g = np.asarray(g, dtype=np.float32).reshape(-1)
    assert np.all(np.isfinite(g)) and np.all(g >= 0), "gains must be finite and non-negative"
    U = g.size
    B = budget_bits(avg_bits, U)
    beta = breakpoints(g)
    vals, inv = np.unique(np.concatenate([beta.reshape(-1), np.zeros(1, np.float32)]), return_inverse=True)
    weight = np.concatenate([np.tile(STEP_BITS, U), [0]])
    per_val = np.bincount(inv.reshape(-1), weights=weight, minlength=vals.size).astype(np.int64)
    above = int(per_val.sum()) - np.cumsum(per_val)      # bits bought strictly above each candidate
    i = int(np.argmax(above <= B))                       # first (smallest) level that fits
    lam = np.float32(vals[i]) + np.float32(0.0)          # canonical +0.0
    return widths_at(beta, lam).astype(np.uint8), lam


def kept_channel_spread(k, bits_tok):
    """sigma_c (R3) of each K channel over the kept prefix tokens of its head; 0 if none kept."""
    k64 = _f64(k)
    Hkv, Np = bits_tok.shape
    out = np.zeros((Hkv, k64.shape[2]))
    for j in range(Hkv):
        kept = np.nonzero(bits_tok[j] > 0)[0]
        if kept.size:
            x = k64[kept, j, :]
            out[j] = np.sqrt(((x - x.mean(axis=0)) ** 2).mean(axis=0))
    return out


def allocate(g_tok, w_chan, k, avg_bits_v, avg_bits_k):
    """Section 2.2 step 2 (V tokens) then step 3 (K channels over the kept tokens), one sequence."""
    Hkv, Np = g_tok.shape
    bits_tok, lam_v = waterfill(g_tok, avg_bits_v)
    bits_tok = bits_tok.reshape(Hkv, Np)
    sig_c = kept_channel_spread(k, bits_tok)
    g_chan = np.asarray(w_chan, np.float32) * sig_c.astype(np.float32)
    bits_chan, lam_k = waterfill(g_chan, avg_bits_k)
    return dict(bits_tok=bits_tok, lam_v=lam_v, sigma_chan=sig_c.astype(np.float32),
                g_chan=g_chan, bits_chan=bits_chan.reshape(g_chan.shape), lam_k=lam_k)


# ---------------------------------------------------------------------------
# Allocation variants (the next rows beside the method: a reading with one
# water level per KV head, and two eviction-only baselines on the same zones)
# ---------------------------------------------------------------------------
def allocate_per_head(g_tok, w_chan, k, avg_bits_v, avg_bits_k):
    """Steps 2 and 3 with one water level per KV head instead of one per sequence:
    each head's V tokens share a budget floor(avg_bits_v * N_p), each head's K channels
    floor(avg_bits_k * D)."""
    Hkv, Np = g_tok.shape
    bits_tok = np.zeros((Hkv, Np), np.uint8)
    lam_v = np.zeros(Hkv, np.float32)
    for j in range(Hkv):
        bits_tok[j], lam_v[j] = waterfill(g_tok[j], avg_bits_v)
    sig_c = kept_channel_spread(k, bits_tok)
    g_chan = np.asarray(w_chan, np.float32) * sig_c.astype(np.float32)
    bits_chan = np.zeros(g_chan.shape, np.uint8)
    lam_k = np.zeros(Hkv, np.float32)
    for j in range(Hkv):
        bits_chan[j], lam_k[j] = waterfill(g_chan[j], avg_bits_k)
    return dict(bits_tok=bits_tok, lam_v=lam_v, sigma_chan=sig_c.astype(np.float32), g_chan=g_chan,
                bits_chan=bits_chan, lam_k=lam_k)


def topk_keep(w, avg_bits):
    """Heavy-hitter eviction (H2O-style): with k = floor(B / 16) tokens affordable at 16 bits
    (B = floor(avg_bits * U)), keep every token whose weight is larger than lambda, the
    smallest non-negative float32 that at most k weights exceed; the others are dropped.
    Written from that definition: sorted descending, lambda is the (k+1)-th value (0 when
    fewer than k+1 weights are positive); equal weights at lambda are all dropped."""
    w = np.asarray(w, dtype=np.float32).reshape(-1)
    assert np.all(np.isfinite(w)) and np.all(w >= 0), "weights must be finite and non-negative"
    kk = budget_bits(avg_bits, w.size) // 16
    srt = np.sort(w)[::-1]
    lam = np.float32(srt[kk]) if kk < w.size and srt[kk] > 0 else np.float32(0.0)
    lam = lam + np.float32(0.0)
    return np.where(w > lam, 16, 0).astype(np.uint8), lam


def threshold_keep(w, tau):
    """Threshold eviction (KVzap-style): keep the tokens whose weight exceeds tau at 16 bits."""
    w = np.asarray(w, dtype=np.float32).reshape(-1)
    return np.where(w > np.float32(tau), 16, 0).astype(np.uint8)


# ---------------------------------------------------------------------------
# TriZone plan and pack (RDKV section 2.3; layout R8)
# ---------------------------------------------------------------------------
KB = 16                                                  # K slots of one k-block


def _ceil_div(a, b):
    return -(-a // b)


def k_slot_in_block(b, i, e):
    """Slot, inside its 16-slot k-block, of element e of the block's word i at K width b
    (project layout; the page fixes no order).  The slots of a block are read in four
    lanes q = 0..3, lane q taking slots 2q, 2q+1 and 2q+8, 2q+9:
      b = 16: word i (of 8) holds slots 2i, 2i+1;
      b = 8:  word i (of 4) holds lane i's slots: 2i, 2i+1 (elements 0, 1) and 2i+8, 2i+9 (2, 3);
      b = 4:  word i (of 2) holds lane 2i's slots (elements 0-3) then lane 2i+1's (4-7),
              each lane's in the order 2q, 2q+1, 2q+8, 2q+9;
      b = 2:  the block's one word holds slots 0..15 in element order."""
    if b == 16:
        return 2 * i + e
    if b == 8:
        return 2 * i + (e % 2) + 8 * (e // 2)
    if b == 4:
        q = 2 * i + e // 4
        return 2 * q + (e % 2) + 8 * ((e // 2) % 2)
    return e


def head_plan(bits_tok_j, bits_chan_j, head_dim):
    """Counts, sizes and orders of one (sequence, KV head).

    K segments (widths 16, 8, 4, 2) hold the channels of their width in ascending
    order, packed into k_words[i] = ceil(n * b / 32) words per token; a segment's
    slot range is whole 16-slot k-blocks (k_blocks[i] of them), the channel of rank
    r going to element r mod (32/b) of word r div (32/b), whose slot follows
    ``k_slot_in_block``; every other slot of the range is a pad (-1).  The K
    quantiser parameters of the 8/4/2-bit slots (meta_slots of them) sit once per
    head in front of its tiles (meta_bytes); a tile holds K codes and, for V width
    b < 16, V codes and V metadata."""
    D = head_dim
    n_v = [int((bits_tok_j == b).sum()) for b in V_CLASSES]
    tiles = [_ceil_div(n, TILE) for n in n_v]
    n_k = [int((bits_chan_j == b).sum()) for b in K_CLASSES]
    k_words = [_ceil_div(n * b, 32) for n, b in zip(n_k, K_CLASSES)]
    k_blocks = [_ceil_div(w * (32 // b), KB) for w, b in zip(k_words, K_CLASSES)]
    row_words = sum(k_words)
    k_slots = KB * sum(k_blocks)
    meta_slots = KB * sum(nb for nb, b in zip(k_blocks, K_CLASSES) if b < 16)
    meta_bytes = 16 * _ceil_div(4 * meta_slots, 16)
    tile_bytes = [4 * TILE * row_words + ((TILE * D * b) // 8 + 4 * D if b < 16 else 0) for b in V_CLASSES]
    slots = []
    for b, nb in zip(K_CLASSES, k_blocks):
        seg = [-1] * (KB * nb)
        per, wpk = 32 // b, b // 2                       # elements per word, words per k-block
        for r, ch in enumerate(np.nonzero(bits_chan_j == b)[0].tolist()):
            wg, e = divmod(r, per)
            seg[KB * (wg // wpk) + k_slot_in_block(b, wg % wpk, e)] = ch
        slots += seg
    tokens = []
    for b, nt in zip(V_CLASSES, tiles):
        t = np.nonzero(bits_tok_j == b)[0].tolist()
        tokens.append(np.array(t + [-1] * (nt * TILE - len(t)), dtype=np.int64))
    return dict(n_v=n_v, tiles=tiles, n_k=n_k + [D - sum(n_k)], k_words=k_words, k_blocks=k_blocks,
                row_words=row_words, k_slots=k_slots, meta_slots=meta_slots, meta_bytes=meta_bytes,
                tile_bytes=tile_bytes,
                a_bytes=meta_bytes + sum(nt * tb for nt, tb in zip(tiles, tile_bytes)),
                slots=np.array(slots, dtype=np.int64), tokens=tokens)


def make_plan(bits_tok, bits_chan, head_dim):
    """Plan of a batch: bits_tok [B, H_kv, N_p], bits_chan [B, H_kv, D]; heads in (b, j) order."""
    B, Hkv = bits_tok.shape[:2]
    heads = []
    a_off = b_row = slot_off = 0
    for b in range(B):
        for j in range(Hkv):
            hp = head_plan(bits_tok[b, j], bits_chan[b, j], head_dim)
            hp.update(a_off=a_off, b_row=b_row, slot_off=slot_off)
            a_off += hp["a_bytes"]
            b_row += TILE * hp["tiles"][3]
            slot_off += TILE * sum(hp["tiles"])
            heads.append(hp)
    present = [(tb, b) for h in heads for tb, nt, b in zip(h["tile_bytes"], h["tiles"], V_CLASSES) if nt]
    return dict(heads=heads, zone_a_bytes=a_off, zone_b_rows=b_row, index_slots=slot_off,
                kept_tokens=int(sum(sum(h["n_v"]) for h in heads)),
                max_tile_bytes=max([tb for tb, b in present] or [0]),
                max_stage_bytes=max([tb + (TILE * head_dim * 2 if b == 16 else 0) for tb, b in present] or [0]))


def quantize_groups(x, b):
    """Asymmetric min-max quantiser ("Solusi 3"): q = round((x - min) / scale),
    scale = (max - min) / (2**b - 1), along the last axis, with fp16 scale and
    zero (R6).  All arithmetic IEEE float32; round half to even; scale 0 -> codes 0.
    Returns codes uint32 (same shape), scale fp16 and zero fp16 (shape without the last axis).
    """
    x = np.asarray(x, dtype=np.float32)
    mn, mx = x.min(axis=-1), x.max(axis=-1)
    zero = mn.astype(np.float16)
    scale = ((mx - mn) / np.float32((1 << b) - 1)).astype(np.float32).astype(np.float16)
    s32 = scale.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        t = (x - zero.astype(np.float32)[..., None]) / s32
    codes = np.clip(np.rint(t), 0, (1 << b) - 1)
    codes = np.where(s32 == 0, 0, codes).astype(np.uint32)
    return codes, scale, zero


def bit_offset(e, b):
    """Bit position of element e (0-based inside its 32-bit word) at width b:
    even elements fill the low half-word, odd elements the high half-word,
    each half LSB-first."""
    return 16 * (e % 2) + b * (e // 2)


def k_word_position(t, w):
    """Index, inside a tile's K words, of word w of token t (0 <= t < 32): the
    words are stored word-major, and inside one word index the tokens sit in
    the order t = 0, 8, 16, 24, 1, 9, 17, 25, ... (position 4 * (t mod 8) + t div 8),
    so tokens t, t+8, t+16, t+24 of one word index are adjacent.  (Project
    layout; the page fixes no byte order.)"""
    return 32 * w + 4 * (t % 8) + t // 8


def v_code_position(p, c, b, head_dim):
    """(word index among a tile's D*b V code words, bit offset) of channel c of token pair p
    (tokens 2p and 2p+1; the odd token's code sits 16 bits above the even one's).  Project
    layout, made for the decode's fragments:
      * pair p = 8 tb + q + 4 h (tb = 16-token block, q = lane of the pair, h = which of the
        lane's two pairs); channel c = 16 cm + 8 s + g (g = lane row, s = which of its two
        row sets); the lane's channel list is k = s * D/16 + cm;
      * lane (g, q) of block tb owns 2 * nw consecutive words (nw = D*b/128), pair h's nw words
        after pair 0's, at ((tb*8 + g)*4 + q) * 2nw + h nw;
      * channel k sits in word k div (16/b) of its pair, at bit b * (k mod (16/b))."""
    D = head_dim
    CM, nw, per = D // 16, D * b // 128, 16 // b
    tb, r = divmod(p, 8)
    q, h = r % 4, r // 4
    cm, rr = divmod(c, 16)
    s, g = divmod(rr, 8)
    k = s * CM + cm
    wk, e = divmod(k, per)
    return ((tb * 8 + g) * 4 + q) * 2 * nw + h * nw + wk, b * e


def v_meta_position(p, grp, head_dim):
    """(index of the 32-bit scale pair, index of the 32-bit zero pair) of token pair p and
    32-channel group grp among a tile's 32*D/32 metadata words; each pair holds the even
    token's fp16 in its low half.  Scales first, ordered (tb, q, h, group), so a lane reads
    every group's scales of its two pairs at once; then zeros, ordered (tb, group, q, h)."""
    NG = head_dim // GROUP
    tb, r = divmod(p, 8)
    q, h = r % 4, r // 4
    return ((tb * 4 + q) * 2 + h) * NG + grp, 16 * NG + ((tb * NG + grp) * 4 + q) * 2 + h


def _k_positions(row_words):
    t = np.arange(TILE)[:, None]
    w = np.arange(row_words)[None, :]
    return k_word_position(t, w)                   # [32, row_words]


def _halves_bits(a):
    return np.asarray(a, dtype=np.float16).view(np.uint16).astype(np.uint32)


def _k_segments(hp):
    """(width, first word, words, first slot, slot list) of each K segment, in row order."""
    seg = []
    w0 = s0 = 0
    for b, nw, nb in zip(K_CLASSES, hp["k_words"], hp["k_blocks"]):
        ns = KB * nb
        seg.append((b, w0, nw, s0, hp["slots"][s0:s0 + ns]))
        w0 += nw
        s0 += ns
    return seg


def _k_word_slots(b, nw):
    """[nw, 32 // b]: the segment slot that element e of the segment's word w holds."""
    per, wpk = 32 // b, b // 2
    return np.array([[KB * (w // wpk) + k_slot_in_block(b, w % wpk, e) for e in range(per)] for w in range(nw)],
                    dtype=np.int64).reshape(nw, per)


def _v_tables(b, head_dim):
    """Word index and bit offset of every (pair, channel) of a V tile: [16, D] each."""
    pos = [[v_code_position(p, c, b, head_dim) for c in range(head_dim)] for p in range(TILE // 2)]
    return (np.array([[x[0] for x in row] for row in pos], dtype=np.int64),
            np.array([[x[1] for x in row] for row in pos], dtype=np.uint64))


def _v_meta_tables(head_dim):
    NG = head_dim // GROUP
    sidx = np.array([[v_meta_position(p, g, head_dim)[0] for g in range(NG)] for p in range(TILE // 2)])
    zidx = np.array([[v_meta_position(p, g, head_dim)[1] for g in range(NG)] for p in range(TILE // 2)])
    return sidx, zidx


def k_head_quantizer(k_j, hp):
    """Per quantised slot of the head (slot order, pads 0): fp16 scale and zero of its channel over
    every kept prefix token of the head (R6: one K group per channel of the head)."""
    kept = np.sort(np.concatenate([t[t >= 0] for t in hp["tokens"]])) if hp["tokens"] else np.zeros(0, np.int64)
    QS = hp["meta_slots"]
    s_q0 = hp["k_slots"] - QS                      # first slot of the 8-bit segment
    ksc = np.zeros(QS, np.float16)
    kze = np.zeros(QS, np.float16)
    for b, _, _, s0, slots in _k_segments(hp):
        if b == 16:
            continue
        for s in np.nonzero(slots >= 0)[0]:
            m = s0 + s - s_q0
            if kept.size:
                _, sc, ze = quantize_groups(k_j[kept, slots[s]], b)
                ksc[m], kze[m] = sc, ze
    return ksc, kze


def pack_head(k_j, v_j, hp, head_dim):
    """Zone-A bytes and zone-B rows of one (sequence, KV head).

    k_j, v_j: [N, D] float32 values of that head.  Layout (little-endian):
      head meta  per quantised K slot (slot order from the first 8-bit slot, pads 0):
                 fp16 scale, fp16 zero of the channel over all kept prefix tokens of the
                 head; padded to meta_bytes (whole 16 bytes)
    then the tiles of each V width in class order:
      K codes    32 rows x row_words uint32 (segments 16, 8, 4, 2 bits, each padded to whole
                 words; element e of a word at bit_offset(e, b) holds the slot given by
                 k_slot_in_block; a 16-bit slot holds the raw fp16 value), word (t, w) stored
                 at k_word_position(t, w)
      V codes    (width b < 16 only) D*b words, channel c of token pair p at v_code_position
      V meta     (b < 16 only) fp16 scale and zero per token and 32-channel group, in pairs of
                 tokens at v_meta_position
    Pad tokens and pad slots hold code 0, scale 0 and zero 0.
    """
    D = head_dim
    out, zone_b = [], []
    seg = _k_segments(hp)
    RW, QS = hp["row_words"], hp["meta_slots"]
    s_q0 = hp["k_slots"] - QS
    ksc, kze = k_head_quantizer(k_j, hp)
    meta = np.zeros(hp["meta_bytes"] // 2, np.float16)
    meta[0:2 * QS:2], meta[1:2 * QS:2] = ksc, kze
    out.append(meta.tobytes())
    NG = D // GROUP
    for ci, bv in enumerate(V_CLASSES):
        toks = hp["tokens"][ci]
        if bv < 16 and hp["tiles"][ci]:
            vword, vbit = _v_tables(bv, D)
            sidx, zidx = _v_meta_tables(D)
        for ti in range(hp["tiles"][ci]):
            tt = toks[ti * TILE:(ti + 1) * TILE]
            real = tt >= 0
            rows = tt[real]
            kw = np.zeros((TILE, RW), dtype=np.uint64)
            for b, wbase, nw, s0, slots in seg:
                if nw == 0:
                    continue
                wslots = _k_word_slots(b, nw)                           # [nw, per]
                codes = np.zeros((rows.size, slots.size), dtype=np.uint64)
                for s in np.nonzero(slots >= 0)[0]:
                    x = k_j[rows, slots[s]]
                    if b == 16:
                        codes[:, s] = _halves_bits(x)
                    else:
                        m = s0 + s - s_q0
                        c, _, _ = quantize_groups_with(x, b, ksc[m], kze[m])
                        codes[:, s] = c
                shifts = np.array([bit_offset(e, b) for e in range(32 // b)], dtype=np.uint64)
                words = (codes[:, wslots] << shifts[None, None, :]).sum(axis=2)    # [real, nw]
                kw[real, wbase:wbase + nw] = words
            kflat = np.zeros(TILE * RW, dtype=np.uint32)
            kflat[_k_positions(RW)] = kw.astype(np.uint32)
            parts = [kflat.tobytes()]
            if bv < 16:
                vals = np.zeros((TILE, D), dtype=np.float32)
                vals[real] = v_j[rows]
                codes, sc, ze = quantize_groups(vals.reshape(TILE, NG, GROUP), bv)
                codes = codes.reshape(TILE, D).astype(np.uint64)
                codes[~real], sc[~real], ze[~real] = 0, 0, 0
                vw = np.zeros(D * bv, dtype=np.uint64)
                np.add.at(vw, vword, (codes[0::2] << vbit) + (codes[1::2] << (vbit + np.uint64(16))))
                vm = np.zeros(2 * 32 * NG, dtype=np.float16)        # 32 * NG 32-bit words as fp16 halves
                vm[2 * sidx], vm[2 * sidx + 1] = sc[0::2], sc[1::2]
                vm[2 * zidx], vm[2 * zidx + 1] = ze[0::2], ze[1::2]
                parts += [vw.astype(np.uint32).tobytes(), vm.tobytes()]
            else:
                rows16 = np.zeros((TILE, D), dtype=np.float16)
                rows16[real] = v_j[rows].astype(np.float16)
                zone_b.append(rows16)
            tile = b"".join(parts)
            assert len(tile) == hp["tile_bytes"][ci]
            out.append(tile)
    zb = np.concatenate(zone_b) if zone_b else np.zeros((0, D), np.float16)
    return b"".join(out), zb


def quantize_groups_with(x, b, scale, zero):
    """Codes of x under given fp16 scale and zero (the quantiser's code rule of
    ``quantize_groups``: IEEE float32 division, round half to even, clamp; scale 0 -> 0)."""
    x = np.asarray(x, dtype=np.float32)
    s32, z32 = np.float32(np.float16(scale)), np.float32(np.float16(zero))
    if s32 == 0:
        return np.zeros(x.shape, np.uint32), scale, zero
    t = (x - z32) / s32
    return np.clip(np.rint(t), 0, (1 << b) - 1).astype(np.uint32), scale, zero


def pack(k, v, bits_tok, bits_chan, window, cap_c=None):
    """TriZone pack of a batch.  k, v [B, N, H_kv, D] (fp16 or fp32).

    Returns dict(plan, zone_a uint8, zone_b fp16 [rows, D], zone_c_k / zone_c_v
    fp16 [B, H_kv, cap_c, D] holding the window in rows [0, W), index int32
    (original position per token slot, -1 for pads), len_c).
    """
    B, N, Hkv, D = k.shape
    plan = make_plan(bits_tok, bits_chan, D)
    cap_c = window if cap_c is None else cap_c
    za, zb = [], []
    index = np.full(plan["index_slots"], -1, dtype=np.int32)
    for hi, hp in enumerate(plan["heads"]):
        b, j = divmod(hi, Hkv)
        a, rows = pack_head(np.asarray(k[b, :, j, :], np.float32), np.asarray(v[b, :, j, :], np.float32), hp, D)
        za.append(a)
        zb.append(rows)
        toks = np.concatenate(hp["tokens"])
        index[hp["slot_off"]:hp["slot_off"] + toks.size] = toks
    zc_k = np.zeros((B, Hkv, cap_c, D), np.float16)
    zc_v = np.zeros((B, Hkv, cap_c, D), np.float16)
    zc_k[:, :, :window] = np.asarray(k[:, N - window:], np.float32).astype(np.float16).transpose(0, 2, 1, 3)
    zc_v[:, :, :window] = np.asarray(v[:, N - window:], np.float32).astype(np.float16).transpose(0, 2, 1, 3)
    return dict(plan=plan, zone_a=np.frombuffer(b"".join(za), dtype=np.uint8).copy(),
                zone_b=np.concatenate(zb) if zb else np.zeros((0, D), np.float16),
                zone_c_k=zc_k, zone_c_v=zc_v, index=index, len_c=window)


def append(cache, k_new, v_new):
    """Zone C receives the fp16 K and V rows of a new token (RDKV section 2.3)."""
    r = cache["len_c"]
    if r >= cache["zone_c_k"].shape[2]:
        raise ValueError("zone C is full")
    cache["zone_c_k"][:, :, r] = np.asarray(k_new, np.float32).astype(np.float16)
    cache["zone_c_v"][:, :, r] = np.asarray(v_new, np.float32).astype(np.float16)
    cache["len_c"] = r + 1


# ---------------------------------------------------------------------------
# Unpack and decode (RDKV section 2.3: attention over zones A, B and C)
# ---------------------------------------------------------------------------
def _field(words, off, b):
    return (words >> np.uint64(off)) & np.uint64((1 << b) - 1)


def unpack_head(zone_a, zone_b, hp, head_dim):
    """Read one head's tiles back: (original positions, K-hat [n, D], V-hat [n, D]) in float64.
    Dequantised value = zero + scale * code; dropped channels read as 0."""
    D = head_dim
    NG = D // GROUP
    RW, QS = hp["row_words"], hp["meta_slots"]
    s_q0 = hp["k_slots"] - QS
    seg = _k_segments(hp)
    toks_all, K_all, V_all = [], [], []
    off = hp["a_off"]
    km = np.frombuffer(zone_a, np.float16, 2 * QS, off).astype(np.float64)
    ksc, kze = km[0::2], km[1::2]
    off += hp["meta_bytes"]
    brow = hp["b_row"]
    for ci, bv in enumerate(V_CLASSES):
        if bv < 16 and hp["tiles"][ci]:
            vword, vbit = _v_tables(bv, D)
            sidx, zidx = _v_meta_tables(D)
        for ti in range(hp["tiles"][ci]):
            tt = hp["tokens"][ci][ti * TILE:(ti + 1) * TILE]
            real = tt >= 0
            kw = np.frombuffer(zone_a, np.uint32, TILE * RW, off)[_k_positions(RW)].astype(np.uint64)   # [32, RW]
            p = off + 4 * TILE * RW
            Kt = np.zeros((TILE, D))
            for b, wbase, nw, s0, slots in seg:
                if nw == 0:
                    continue
                wslots = _k_word_slots(b, nw)
                for w in range(nw):
                    for e in range(32 // b):
                        s = wslots[w, e]
                        ch = slots[s]
                        if ch < 0:
                            continue
                        code = _field(kw[:, wbase + w], bit_offset(e, b), b)
                        if b == 16:
                            Kt[:, ch] = code.astype(np.uint16).view(np.float16).astype(np.float64)
                        else:
                            m = s0 + s - s_q0
                            Kt[:, ch] = kze[m] + ksc[m] * code.astype(np.float64)
            if bv < 16:
                vw = np.frombuffer(zone_a, np.uint32, D * bv, p).astype(np.uint64)
                p += 4 * vw.size
                vm = np.frombuffer(zone_a, np.float16, 2 * 32 * NG, p).astype(np.float64)
                p += 2 * vm.size
                Vt = np.zeros((TILE, D))
                for par in range(2):            # even, odd token of each pair
                    code = _field(vw[vword], vbit + np.uint64(16 * par), bv).astype(np.float64)   # [16, D]
                    sc = vm[2 * sidx + par]                                                      # [16, NG]
                    ze = vm[2 * zidx + par]
                    Vt[par::2] = np.repeat(ze, GROUP, axis=1) + np.repeat(sc, GROUP, axis=1) * code
            else:
                Vt = zone_b[brow:brow + TILE].astype(np.float64)
                brow += TILE
            assert p - off == hp["tile_bytes"][ci]
            off = p
            toks_all.append(tt[real])
            K_all.append(Kt[real])
            V_all.append(Vt[real])
    if not toks_all:
        return np.zeros(0, np.int64), np.zeros((0, D)), np.zeros((0, D))
    return np.concatenate(toks_all), np.concatenate(K_all), np.concatenate(V_all)


def attention(q, K, V):
    """Textbook softmax attention of one query over rows K, V (scale 1/sqrt(D)), float64.
    With no rows the output is 0."""
    q = _f64(q)
    if K.shape[0] == 0:
        return np.zeros(q.shape[-1])
    s = _f64(K) @ q / math.sqrt(q.shape[-1])
    p = np.exp(s - s.max())
    p /= p.sum()
    return p @ _f64(V)


def unpack(cache, head_dim):
    """Per head: (positions, K-hat, V-hat) of zones A and B."""
    return [unpack_head(cache["zone_a"].tobytes(), cache["zone_b"], hp, head_dim) for hp in cache["plan"]["heads"]]


def decode(cache, q, unpacked=None):
    """One decode step: out [B, H_q, D] float64 attending over zones A+B of the
    plan and rows [0, len_c) of zone C, for queries q [B, H_q, D]."""
    q64 = _f64(q)
    B, Hq, D = q64.shape
    Hkv = cache["zone_c_k"].shape[1]
    G = Hq // Hkv
    un = unpacked if unpacked is not None else unpack(cache, D)
    L = cache["len_c"]
    out = np.zeros((B, Hq, D))
    for b in range(B):
        for j in range(Hkv):
            _, Ka, Va = un[b * Hkv + j]
            K = np.concatenate([Ka, cache["zone_c_k"][b, j, :L].astype(np.float64)])
            V = np.concatenate([Va, cache["zone_c_v"][b, j, :L].astype(np.float64)])
            for h in range(j * G, (j + 1) * G):
                out[b, h] = attention(q64[b, h], K, V)
    return out


def decode_bytes(plan, head_dim, h_q, h_kv, len_c, batch):
    """Algorithmic bytes one decode step must read and write: zone-A payload and
    metadata of real tokens and real channels (the K metadata once per head),
    zone-B rows of real tokens, zone-C rows, q (fp16) and out (fp32).  Padding is
    excluded."""
    D = head_dim
    total = 0
    for hp in plan["heads"]:
        n16k, n8k, n4k, n2k, _ = hp["n_k"]
        kq = n8k + n4k + n2k
        ntok = sum(hp["n_v"])
        k_payload = ntok * (2 * n16k + (8 * n8k + 4 * n4k + 2 * n2k) / 8)
        k_meta = 4 * kq if ntok else 0                  # scale and zero per quantised channel, once per head
        v_payload = sum(n * (D * b / 8 + (4 * D / GROUP if b < 16 else 0)) for n, b in zip(hp["n_v"], V_CLASSES))
        total += k_payload + k_meta + v_payload + len_c * 4 * D
    total += batch * h_q * D * (2 + 4)
    return total


# ---------------------------------------------------------------------------
# Zone-C re-compression (next row beside the method).  New tokens start in
# zone C at fp16 (RDKV section 2.3); the pages do not say how they later join
# zones A and B.  Reading R10 (a project decision):
#  * the oldest rows of zone C (all but a recent tail) move into a new segment,
#    a TriZone cache of their own with no window;
#  * their token weights are the attention the recent decode queries gave
#    them: w_t = (N / R) * sum over the R recent queries tau and the G heads
#    of the group of exp(q.k_t / sqrt(D) - lse_tau,h), lse the log-sum-exp of
#    that decode; a prefill weight sums the attention of up to N query rows,
#    and the factor puts the moved tokens on that scale; sigma_t and g_t as in
#    step 1;
#  * the allocation is incremental: the instance keeps its water levels
#    lambda_V, lambda_K of the prefill and the moved units take the Lagrangian
#    choice at those levels (section 2.2), K channels over the moved kept
#    tokens with the prefill's channel weights w_c;
#  * the attention over several segments and the live zone C is the softmax
#    over the union of their keys, merged from each part's output and
#    log-sum-exp.
# ---------------------------------------------------------------------------
def attention_lse(q, K, V):
    """attention(q, K, V) and its log-sum-exp ln sum_t exp(q . k_t / sqrt(D)); -inf with no rows."""
    q = _f64(q)
    if K.shape[0] == 0:
        return np.zeros(q.shape[-1]), -np.inf
    s = _f64(K) @ q / math.sqrt(q.shape[-1])
    m = s.max()
    e = np.exp(s - m)
    return (e @ _f64(V)) / e.sum(), m + math.log(e.sum())


def decode_lse(cache, q, unpacked=None):
    """decode() and the log-sum-exp of every query head: (out [B, H_q, D], lse [B, H_q]) float64."""
    q64 = _f64(q)
    B, Hq, D = q64.shape
    Hkv = cache["zone_c_k"].shape[1]
    G = Hq // Hkv
    un = unpacked if unpacked is not None else unpack(cache, D)
    L = cache["len_c"]
    out, lse = np.zeros((B, Hq, D)), np.full((B, Hq), -np.inf)
    for b in range(B):
        for j in range(Hkv):
            _, Ka, Va = un[b * Hkv + j]
            K = np.concatenate([Ka, cache["zone_c_k"][b, j, :L].astype(np.float64)])
            V = np.concatenate([Va, cache["zone_c_v"][b, j, :L].astype(np.float64)])
            for h in range(j * G, (j + 1) * G):
                out[b, h], lse[b, h] = attention_lse(q64[b, h], K, V)
    return out, lse


def merge_attention(outs, lses):
    """Attention over the union of disjoint key sets from each part's output and log-sum-exp:
    out = sum_i e^(lse_i) out_i / sum_i e^(lse_i), lse = ln sum_i e^(lse_i).
    outs [P, ..., D], lses [P, ...]; parts without keys (lse = -inf) weigh 0; no keys at all: 0, -inf."""
    outs, lses = _f64(outs), _f64(lses)
    m = lses.max(axis=0)
    safe = np.where(np.isfinite(m), m, 0.0)
    wts = np.where(np.isfinite(lses), np.exp(lses - safe[None]), 0.0)
    tot = wts.sum(axis=0)
    out = np.where(tot[..., None] > 0, (wts[..., None] * outs).sum(axis=0) / np.where(tot > 0, tot, 1.0)[..., None],
                   0.0)
    lse = np.where(tot > 0, safe + np.log(np.where(tot > 0, tot, 1.0)), -np.inf)
    return out, lse


def take_zone_c(cache, n_move):
    """Removes rows [0, n_move) of zone C: returns them as k, v [B, n_move, H_kv, D] (fp16 values)
    and moves rows [n_move, len_c) to the front."""
    L = cache["len_c"]
    if not 0 < n_move <= L:
        raise ValueError("n_move outside (0, len_c]")
    k = cache["zone_c_k"][:, :, :n_move].transpose(0, 2, 1, 3).copy()
    v = cache["zone_c_v"][:, :, :n_move].transpose(0, 2, 1, 3).copy()
    rest = L - n_move
    cache["zone_c_k"][:, :, :rest] = cache["zone_c_k"][:, :, n_move:L].copy()
    cache["zone_c_v"][:, :, :rest] = cache["zone_c_v"][:, :, n_move:L].copy()
    cache["len_c"] = rest
    return k, v


def recent_token_weights(k_seg, q_recent, lse_recent, scale=1.0):
    """R10 token weights of moved tokens.  k_seg [n, H_kv, D], q_recent [R, H_q, D], lse_recent
    [R, H_q] (natural log) -> w [H_kv, n] float64: sum over the R queries and the G heads of the
    group of exp(q . k_t / sqrt(D) - lse), times `scale` (N / R: the prefill's weights sum over up to
    N query rows)."""
    k64, q64, l64 = _f64(k_seg), _f64(q_recent), _f64(lse_recent)
    n, Hkv, D = k64.shape
    R, Hq, _ = q64.shape
    G = Hq // Hkv
    w = np.zeros((Hkv, n))
    for h in range(Hq):
        j = h // G
        s = q64[:, h, :] @ k64[:, j, :].T / math.sqrt(D)       # [R, n]
        w[j] += np.exp(s - l64[:, h][:, None]).sum(axis=0)
    return w * scale


def recompress_gains(k_seg, v_seg, q_recent, lse_recent, scale=1.0):
    """R10 step 1 for the moved tokens of one sequence: w_tok, sigma_tok (float32) and g_tok."""
    w = recent_token_weights(k_seg, q_recent, lse_recent, scale)
    sig = value_spread(v_seg)
    n = k_seg.shape[0]
    return dict(w_tok=w.astype(np.float32), sigma_tok=sig.astype(np.float32), g_tok=token_gains(w, sig, n))


def allocate_at_levels(g_tok, w_chan, k, lam_v, lam_k):
    """R10 incremental allocation of one sequence: V widths at water level lam_v, then sigma_c over
    the kept moved tokens, g_c = fl32(w_c * sigma_c) and K widths at lam_k (section 2.2 steps 2-3
    with the levels given instead of found)."""
    g_tok = np.asarray(g_tok, np.float32)
    Hkv, n = g_tok.shape
    bits_tok = widths_at(breakpoints(g_tok), lam_v).astype(np.uint8).reshape(Hkv, n)
    sig_c = kept_channel_spread(k, bits_tok)
    g_chan = np.asarray(w_chan, np.float32) * sig_c.astype(np.float32)
    bits_chan = widths_at(breakpoints(g_chan), lam_k).astype(np.uint8).reshape(g_chan.shape)
    return dict(bits_tok=bits_tok, sigma_chan=sig_c.astype(np.float32), g_chan=g_chan, bits_chan=bits_chan)
