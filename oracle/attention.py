"""fp64 oracle: exact softmax attention and its (m, l, O) triplet algebra.

TEST INFRASTRUCTURE ONLY (see the package docstring): the product path never
imports this module.

Conventions shared with the library's C-ABI (token-major layouts):
  q, o            [B, S_q, h_q, D]
  k, v            [B, S_kv, h_kv, D]
  lse, m, l       [B, h_q, S_q]
  unnormalised O  [B, S_q, h_q, D]
  stacked partials: a leading chunk axis C in front of each of the above.
Query i sits at absolute position q_pos0 + i, key j at position kv_pos0 + j.
Under causal masking key j is visible to query i iff its position is <= the
query's (top-left alignment: the same index space for Q and KV, as in the
dependent inner-loop end min(kv_end, tile_q.end) of "[pallas] Support dependent
Tile.end bounds in Pallas", opening example).  Query head h reads KV head
floor(h / G), G = h_q / h_kv (contiguous head groups).
Sliding window (optional, causal only): key j is visible to query i iff
pos(i) - window <= pos(j) <= pos(i), i.e. the `window` keys before the query and
the query's own.  This is the dependent lower bound max(kv_begin, tile_q.begin -
window) that "[pallas] Support dependent Tile.end bounds in Pallas" ("Scalar
minimum") defers to sliding-window support, taken at element level.

Sources (page title, section):
  * "kernbench2 _gqa_prefill_long.py", gqa_prefill_long_kernel:
    step 0 computes scores = Q.K^T, m = rowmax, exp(scores - m), l = rowsum,
    O = exp_scores . V (unnormalised); steps 1..C-1 merge each step into the
    running triplet with m_new = max(m, m_step) and the two exp(m - m_new)
    factors; the final step divides O by l.
  * "kernbench2 _attention_mesh_mlo.py": the one-shot local partial of a
    sequence shard, the same pairwise merge (merge-from-W / merge-from-E) and
    the final normalisation O := o / l.
Readings where the pages are silent or garbled: the softmax scale is applied
to the scores before the max (the prefill page omits it); K is transposed
(the prefill page's reshape is only right for zero or symmetric inputs); the
decode page's softmax-normalised `o` is read as the unnormalised sum that its
merge and final division require; a fully masked row or empty range is the
merge identity (m, l, O) = (-inf, 0, 0) and yields O = 0, LSE = -inf.
"""

from __future__ import annotations

import math

import numpy as np

NEG_INF = -np.inf


def _f64(x) -> np.ndarray:
    """Host fp64 copy of an array or a (CPU) torch tensor."""
    if hasattr(x, "detach"):
        x = x.detach().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def _kv_head(h: int, group: int) -> int:
    """KV head read by query head h: contiguous groups of `group` query heads."""
    return h // group


def _visible(q_pos: np.ndarray, k_pos: np.ndarray, causal: bool, window: int | None = None) -> np.ndarray:
    """[len(q_pos), len(k_pos)] visibility: all pairs, or key position <= query position,
    and with a window also key position >= query position - window."""
    if not causal:
        if window is not None:
            raise ValueError("a sliding window needs causal masking")
        return np.ones((q_pos.size, k_pos.size), dtype=bool)
    vis = k_pos[None, :] <= q_pos[:, None]
    if window is not None:
        if window < 0:
            raise ValueError("window must be >= 0")
        vis &= k_pos[None, :] >= q_pos[:, None] - window
    return vis


def _scores(q_rows: np.ndarray, k_rows: np.ndarray, scale: float) -> np.ndarray:
    """s_ij = scale * sum_d q[i, d] * k[j, d]   (Q . K^T, scale before the max)."""
    return scale * (q_rows @ k_rows.T)


def _row_triplet(s: np.ndarray, vis: np.ndarray, v_rows: np.ndarray):
    """Partial triplet of one KV range for a block of query rows.

    m = max over visible keys of s; l = sum exp(s - m); O = sum exp(s - m) v.
    Rows with no visible key give the identity (-inf, 0, 0).
    """
    s = np.where(vis, s, NEG_INF)
    m = s.max(axis=1) if s.shape[1] else np.full(s.shape[0], NEG_INF)
    finite = np.isfinite(m)
    shift = np.where(finite, m, 0.0)
    p = np.where(vis, np.exp(s - shift[:, None]), 0.0)
    l = p.sum(axis=1)
    o = p @ v_rows
    m = np.where(finite, m, NEG_INF)
    return m, l, o


def attention(q, k, v, scale: float, causal: bool = False, q_pos0: int = 0,
              kv_pos0: int = 0, rows=None, heads=None, batches=None, window: int | None = None):
    """Exact softmax attention, written out from its definition.

    O_i = sum_j softmax_j(s_i) v_j over the visible keys j, LSE_i = ln sum_j e^{s_ij}.
    `rows`, `heads`, `batches` optionally restrict which outputs are computed
    (sampled checks at large sizes); every computed row still reads every key.
    Returns (O [B, S_q, h_q, D], LSE [B, h_q, S_q]) in fp64; rows not computed
    are NaN.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, S_q, h_q, D = q.shape
    _, S_kv, h_kv, _ = k.shape
    if h_q % h_kv:
        raise ValueError("h_q must be a multiple of h_kv")
    group = h_q // h_kv
    rows = np.arange(S_q) if rows is None else np.asarray(rows, dtype=np.int64)
    heads = range(h_q) if heads is None else heads
    batches = range(B) if batches is None else batches
    out = np.full((B, S_q, h_q, v.shape[-1]), np.nan)
    lse = np.full((B, h_q, S_q), np.nan)
    vis = _visible(q_pos0 + rows, kv_pos0 + np.arange(S_kv), causal, window)
    for b in batches:
        for h in heads:
            g = _kv_head(h, group)
            s = _scores(q[b, rows, h, :], k[b, :, g, :], scale)
            m, l, o = _row_triplet(s, vis, v[b, :, g, :])
            has = l > 0
            out[b, rows, h, :] = np.where(has[:, None], o / np.where(has, l, 1.0)[:, None], 0.0)
            lse[b, h, rows] = np.where(has, m + np.log(np.where(has, l, 1.0)), NEG_INF)
    return out, lse


def partial(q, k, v, scale: float, causal: bool = False, q_pos0: int = 0,
            kv_begin: int = 0, kv_end: int | None = None):
    """One KV range's partial triplet: the prefill page's per-step partial.

    Keys are k[:, kv_begin:kv_end] at positions kv_begin.. (the index space of
    k), queries at q_pos0 + i.  Returns m, l [B, h_q, S_q] and the
    unnormalised O [B, S_q, h_q, D] in fp64.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, S_q, h_q, D = q.shape
    S_kv, h_kv = k.shape[1], k.shape[2]
    kv_end = S_kv if kv_end is None else kv_end
    group = h_q // h_kv
    keys = np.arange(kv_begin, kv_end)
    vis = _visible(q_pos0 + np.arange(S_q), keys, causal)
    m = np.empty((B, h_q, S_q))
    l = np.empty((B, h_q, S_q))
    o = np.empty((B, S_q, h_q, v.shape[-1]))
    for b in range(B):
        for h in range(h_q):
            g = _kv_head(h, group)
            s = _scores(q[b, :, h, :], k[b, keys, g, :], scale)
            m[b, h], l[b, h], o[b, :, h, :] = _row_triplet(s, vis, v[b, keys, g, :])
    return m, l, o


def _merge_pair(m, l, o, m_s, l_s, o_s):
    """Fold triplet (m_s, l_s, o_s) into the running (m, l, o).

    m_new = max(m, m_s); scale_old = exp(m - m_new); scale_step = exp(m_s - m_new);
    l_new = l*scale_old + l_s*scale_step; o_new = o*scale_old + o_s*scale_step.
    When m_new = -inf (both sides empty) both factors are 0, not NaN.
    m, l have shape R, o has shape R + (D,).
    """
    m_new = np.maximum(m, m_s)
    finite = np.isfinite(m_new)
    ref = np.where(finite, m_new, 0.0)
    scale_old = np.where(finite, np.exp(m - ref), 0.0)
    scale_step = np.where(finite, np.exp(m_s - ref), 0.0)
    l_new = l * scale_old + l_s * scale_step
    o_new = o * scale_old[..., None] + o_s * scale_step[..., None]
    return m_new, l_new, o_new


def merge(ms, ls, os_, order=None):
    """Fold C stacked partials with the pairwise merge, then normalise.

    ms, ls: [C, B, H, S]; os_: [C, B, S, H, D] (the library's partial layout).
    `order` optionally permutes the fold order (the result is order-free up
    to rounding).  Returns (O [B, S, H, D], LSE [B, H, S]); a row whose
    partials are all empty gives O = 0 and LSE = -inf.
    """
    ms, ls, os_ = _f64(ms), _f64(ls), _f64(os_)
    order = range(ms.shape[0]) if order is None else order
    order = list(order)
    # work in [B, H, S] row order: move O's head axis in front of S
    o_rows = np.swapaxes(os_, 2, 3)  # [C, B, H, S, D]
    first = order[0]
    m, l, o = ms[first], ls[first], o_rows[first]
    for c in order[1:]:
        m, l, o = _merge_pair(m, l, o, ms[c], ls[c], o_rows[c])
    has = l > 0
    safe_l = np.where(has, l, 1.0)
    out = np.where(has[..., None], o / safe_l[..., None], 0.0)
    lse = np.where(has, m + np.log(safe_l), NEG_INF)
    return np.swapaxes(out, 1, 2), lse


def chunk_bounds(length: int, num_chunks: int):
    """Split [0, length) into num_chunks ranges of ceil(length / num_chunks) keys.

    Trailing chunks may be short or empty (empty ones contribute the identity).
    """
    step = -(-length // num_chunks)
    return [(min(c * step, length), min((c + 1) * step, length)) for c in range(num_chunks)]


def ring_prefill(q, k, v, scale: float, causal: bool, num_chunks: int):
    """The prefill page's ring algorithm on one device: a partial per KV chunk,
    merged in ring order starting at each query block's own chunk.

    For query block r (the rows sharing chunk r's positions) the chunks are
    visited (r + t) mod C, t = 0..C-1, exactly as a CUBE that starts on its own
    block and receives from its east neighbour.  Returns (O, LSE) like
    `attention`; equals it up to rounding.
    """
    q = _f64(q)
    B, S_q, h_q, D = q.shape
    S_kv = _f64(k).shape[1]
    bounds = chunk_bounds(S_kv, num_chunks)
    step = -(-S_kv // num_chunks)
    out = np.empty((B, S_q, h_q, _f64(v).shape[-1]))
    lse = np.empty((B, h_q, S_q))
    parts = [partial(q, k, v, scale, causal, 0, lo, hi) for lo, hi in bounds]
    ms = np.stack([p[0] for p in parts])
    ls = np.stack([p[1] for p in parts])
    os_ = np.stack([p[2] for p in parts])
    for i in range(S_q):
        r = min(i // step, num_chunks - 1)
        order = [(r + t) % num_chunks for t in range(num_chunks)]
        o_i, lse_i = merge(ms[:, :, :, i:i + 1], ls[:, :, :, i:i + 1], os_[:, :, i:i + 1], order)
        out[:, i] = o_i[:, 0]
        lse[:, :, i] = lse_i[:, :, 0]
    return out, lse


def jagged_attention(q, k, v, seq_offsets, scale: float, causal: bool = True,
                     seqs=None, heads=None):
    """Variable-length self-attention over packed sequences.

    q, k, v: [T, H, D]; sequence b spans tokens [seq_offsets[b], seq_offsets[b+1])
    and attends only within itself (the jagged KV end seq_offsets[seq_idx + 1]).
    Returns (O [T, H, D], LSE [H, T]); tokens of sequences not in `seqs` are NaN.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    offs = np.asarray(seq_offsets, dtype=np.int64)
    T, H, D = q.shape
    out = np.full((T, H, v.shape[-1]), np.nan)
    lse = np.full((H, T), np.nan)
    seqs = range(offs.size - 1) if seqs is None else seqs
    for b in seqs:
        lo, hi = int(offs[b]), int(offs[b + 1])
        if hi == lo:
            continue
        o_b, lse_b = attention(q[None, lo:hi], k[None, lo:hi], v[None, lo:hi], scale, causal,
                               heads=heads)
        out[lo:hi] = o_b[0]
        lse[:, lo:hi] = lse_b[0]
    return out, lse


def decode_partials(q, k, v, scale: float, num_splits: int, batches=None, heads=None):
    """Split-KV decode partials: one one-shot local partial per KV chunk.

    q: [B, h_q, D] (one query per sequence); k, v: [B, S_kv, h_kv, D].
    Returns stacked m, l [C, B, h_q] and unnormalised O [C, B, h_q, D] (fp64);
    batch/head entries outside `batches`/`heads` are NaN.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, h_q, D = q.shape
    S_kv, h_kv = k.shape[1], k.shape[2]
    group = h_q // h_kv
    batches = range(B) if batches is None else batches
    heads = range(h_q) if heads is None else heads
    bounds = chunk_bounds(S_kv, num_splits)
    m = np.full((num_splits, B, h_q), np.nan)
    l = np.full((num_splits, B, h_q), np.nan)
    o = np.full((num_splits, B, h_q, v.shape[-1]), np.nan)
    for b in batches:
        for h in heads:
            g = _kv_head(h, group)
            for c, (lo, hi) in enumerate(bounds):
                keys = np.arange(lo, hi)
                s = _scores(q[b, h][None, :], k[b, keys, g, :], scale)
                vis = np.ones((1, keys.size), dtype=bool)
                mm, ll, oo = _row_triplet(s, vis, v[b, keys, g, :])
                m[c, b, h], l[c, b, h], o[c, b, h] = mm[0], ll[0], oo[0]
    return m, l, o


def decode(q, k, v, scale: float, num_splits: int, batches=None, heads=None):
    """Split-KV decode result: decode_partials folded by `merge`.

    Returns (O [B, h_q, D], LSE [B, h_q]).
    """
    m, l, o = decode_partials(q, k, v, scale, num_splits, batches, heads)
    # partial layout with S_q = 1: m,l [C,B,H,1], O [C,B,1,H,D]
    out, lse = merge(m[..., None], l[..., None], o[:, :, None])
    return out[:, 0], lse[..., 0]


def causal_useful_flops(lengths_q_kv, head_dim: int, heads: int, causal: bool = True) -> float:
    """4 * D * H * (number of visible (query, key) pairs), summed over sequences.

    lengths_q_kv: iterable of (S_q, S_kv) per sequence, top-left aligned.
    Causal with S_q = S_kv = L contributes L(L+1)/2 pairs.
    """
    pairs = 0
    for s_q, s_kv in lengths_q_kv:
        if causal:
            pairs += sum(min(i + 1, s_kv) for i in range(s_q)) if s_q != s_kv else s_q * (s_q + 1) // 2
        else:
            pairs += s_q * s_kv
    return 4.0 * head_dim * heads * pairs


def window_useful_flops(length: int, window: int, head_dim: int, heads: int) -> float:
    """4 * D * H * (visible pairs) of one causal sequence under a sliding window:
    query i sees min(i, window) + 1 keys."""
    pairs = sum(min(i, window) + 1 for i in range(length))
    return 4.0 * head_dim * heads * pairs


def log_sum_exp_uniform(n: int) -> float:
    """LSE of n equal zero scores: ln n."""
    return math.log(n)
