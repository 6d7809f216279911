"""Plain fp64 attention: the definition, forward and backward, and the
conditional-rescale online-softmax algorithm restated step by step.

TEST INFRASTRUCTURE ONLY (see the package docstring): imported by tests, the
smoke check and the benchmark's CPU baseline, never by the product path.

Sources
-------
* Exact attention, tiled with an online softmax, computes the same result as
  materialising softmax(scale * Q K^T) and multiplying by V:
  ainexis deep-dive "Tri Dao FlashAttention-4", section 背景 (first stage:
  tiling + online softmax) and section 横向扩展, concept 2 (online softmax keeps
  a running max and running sum and corrects earlier partial results).
* Conditional rescaling: rescale only when the new tile's row max exceeds the
  running max by more than a threshold of 8.0 (a factor 2^8 = 256), with a final
  exact normalisation: wittx "FlashAttention-4", section 90%的rescaling都是白干的;
  jsqmd "GPU 算力翻倍…FlashAttention-4", section 四.3.
* Backward (dQ, dK, dV for the loss <O, dO>), including the dQ reduction over
  the key dimension: wittx "FlashAttention-4", section 反向传播的优化. The pages
  give no formulas; the gradients below are the calculus of the definition.
* Score modifications (FlexAttention variants built on FA4: wittx
  "FlashAttention-4", section Python写GPU内核; newton wiki "FlashAttention-4",
  發展歷程). The pages name FlexAttention but no modification; the two below
  are its standard examples, applied to the scaled logit a_ij before the mask
  and the softmax (see :func:`score_mod_apply`).

Conventions (readings where the pages are silent)
-------------------------------------------------
* One head at a time: q [Nq, d_qk], k [Nk, d_qk], v [Nk, d_v], do [Nq, d_v].
* Causal mask is bottom-right aligned: key j is visible to query i iff
  j <= i + (Nk - Nq). With Nq == Nk this is j <= i.
* A row with no visible key has O = 0, LSE = -inf and zero gradients.
* LSE is the natural-log logsumexp of the scaled logits.
* Inputs are taken exactly as given (bf16 values upcast exactly to fp64).
"""

from __future__ import annotations

import math

import numpy as np

LN2 = math.log(2.0)
LOG2E = 1.0 / LN2


def _f64(a) -> np.ndarray:
    if hasattr(a, "detach"):  # torch tensor (CPU) → numpy, exact upcast
        a = a.detach().to("cpu").double().numpy()
    return np.asarray(a, dtype=np.float64)


def visible_limit(i, nq: int, nk: int, causal: bool):
    """Number of visible keys for query row(s) i: keys 0 .. limit-1 are visible."""
    i = np.asarray(i)
    if not causal:
        return np.full(i.shape, nk, dtype=np.int64)
    return np.clip(i + (nk - nq) + 1, 0, nk).astype(np.int64)


def _logits(q, k, softmax_scale, rows, nq, nk, causal, visible=None, score_mod=None, with_deriv=False):
    """a_ij = mod(scale * q_i . k_j) for visible j, -inf elsewhere (rows = row indices).
    ``visible`` (optional bool [Nq, Nk]) hides further keys (AND with the causal mask);
    ``score_mod`` as in :func:`score_mod_apply`. With ``with_deriv`` also returns
    the modification's derivative."""
    a, da = score_mod_apply(softmax_scale * (q[rows] @ k.T), rows, nq, nk, score_mod)
    lim = visible_limit(rows, nq, nk, causal)
    cols = np.arange(nk)
    a[cols[None, :] >= lim[:, None]] = -np.inf
    if visible is not None:
        a[~np.asarray(visible, dtype=bool)[rows]] = -np.inf
    return (a, da) if with_deriv else a


def score_mod_apply(a, rows, nq: int, nk: int, score_mod):
    """A score modification of the scaled logits a = scale * q_i . k_j (rows:
    the query indices of a's rows; all nk keys as columns).

    * ``None``: a unchanged.
    * ``("softcap", c)``, c > 0: a' = c * tanh(a / c) (logits soft-capped to (-c, c)).
    * ``("alibi", m)``, m >= 0: a' = a - m * |j - (i + nk - nq)|, a linear penalty on the
      distance between key j and query i, with the query's position aligned
      bottom-right like the causal mask.

    Returns (a', da'/da), the derivative elementwise (1 for the additive bias).
    """
    if score_mod is None:
        return a, np.ones_like(a)
    kind, val = score_mod
    if kind == "softcap":
        c = float(val)
        t = np.tanh(a / c)
        return c * t, 1.0 - t * t
    if kind == "alibi":
        qpos = np.asarray(rows)[:, None] + (nk - nq)
        dist = np.abs(np.arange(nk)[None, :] - qpos)
        return a - float(val) * dist, np.ones_like(a)
    raise ValueError(f"unknown score modification {kind!r}")


def block_sparse_visible(nq: int, nk: int, kv_count, kv_index, q_block: int = 256, k_block: int = 128):
    """Key visibility of a block-sparse mask, written out element by element.

    The mask lists, for each block of ``q_block`` query rows, the blocks of
    ``k_block`` keys it attends to: query block b sees key blocks
    kv_index[b, 0 .. kv_count[b]-1] (FlexAttention / block-sparse variants
    built on FA4: wittx "FlashAttention-4", section Python写GPU内核). Entries
    outside [0, ceil(nk / k_block)) list nothing. Returns bool [nq, nk].
    """
    kv_count = np.asarray(kv_count).reshape(-1)
    kv_index = np.asarray(kv_index)
    vis = np.zeros((nq, nk), dtype=bool)
    for i in range(nq):
        b = i // q_block
        n = int(kv_count[b]) if b < kv_count.shape[0] else 0
        for t in range(max(0, min(n, kv_index.shape[1] if kv_index.ndim == 2 else 0))):
            kb = int(kv_index[b, t])
            if 0 <= kb and kb * k_block < nk:
                vis[i, kb * k_block:min(nk, (kb + 1) * k_block)] = True
    return vis


def _row_blocks(nq: int, row_block):
    rb = nq if not row_block else int(row_block)
    rb = max(rb, 1)
    for r0 in range(0, nq, rb):
        yield np.arange(r0, min(nq, r0 + rb))


def attention_fwd(q, k, v, softmax_scale: float, causal: bool = False, row_block=None, visible=None,
                  score_mod=None):
    """Dense definition of one head's forward pass.

    O_i = sum_j softmax_j(a_i) v_j with a_ij = scale * q_i . k_j (masked → -inf),
    LSE_i = log sum_j exp(a_ij). Computed as: m_i = max_j a_ij,
    l_i = sum_j exp(a_ij - m_i), O_i = (sum_j exp(a_ij - m_i) v_j) / l_i,
    LSE_i = m_i + log l_i.  ``row_block`` only bounds memory: rows are
    independent, each row is still computed over all of its keys at once.
    ``visible`` (bool [Nq, Nk], optional) masks further keys, e.g. a block-
    sparse mask from :func:`block_sparse_visible`. ``score_mod`` replaces a_ij
    by its modification (:func:`score_mod_apply`) before the mask.

    Returns (O [Nq, d_v], LSE [Nq]) in fp64.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    nq, nk, dv = q.shape[0], k.shape[0], v.shape[1]
    o = np.zeros((nq, dv))
    lse = np.full(nq, -np.inf)
    if nq == 0 or nk == 0:
        return o, lse
    for rows in _row_blocks(nq, row_block):
        a = _logits(q, k, softmax_scale, rows, nq, nk, causal, visible, score_mod)
        m = a.max(axis=1)
        live = np.isfinite(m)
        if not live.any():
            continue
        e = np.exp(a[live] - m[live, None])
        l = e.sum(axis=1)
        o[rows[live]] = (e @ v) / l[:, None]
        lse[rows[live]] = m[live] + np.log(l)
    return o, lse


def attention_bwd(q, k, v, do, softmax_scale: float, causal: bool = False, row_block=None, visible=None,
                  score_mod=None):
    """Dense definition of one head's backward pass for the loss <O, dO>.

    P_ij = exp(a_ij - LSE_i); dV_j = sum_i P_ij dO_i; dP_ij = dO_i . v_j;
    D_i = sum_j P_ij dP_ij; dS_ij = P_ij (dP_ij - D_i) * a'_ij, a' the derivative
    of the score modification (1 without one);
    dQ_i = scale * sum_j dS_ij k_j; dK_j = scale * sum_i dS_ij q_i.
    ``visible`` masks further keys as in :func:`attention_fwd` (P_ij = 0 there).

    Returns dict with dq, dk, dv (fp64) and D (the row term, computed as
    sum_j P_ij dP_ij so that tests can check it against dO_i . O_i).
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    nq, nk = q.shape[0], k.shape[0]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    D = np.zeros(nq)
    if nq == 0 or nk == 0:
        return {"dq": dq, "dk": dk, "dv": dv, "D": D}
    for rows in _row_blocks(nq, row_block):
        a, da = _logits(q, k, softmax_scale, rows, nq, nk, causal, visible, score_mod, with_deriv=True)
        m = a.max(axis=1)
        live = np.isfinite(m)
        if not live.any():
            continue
        rl = rows[live]
        al = a[live]
        lse = m[live] + np.log(np.exp(al - m[live, None]).sum(axis=1))
        p = np.exp(al - lse[:, None])
        dv += p.T @ do[rl]
        dp = do[rl] @ v.T
        d_row = (p * dp).sum(axis=1)
        ds = p * (dp - d_row[:, None]) * da[live]
        dq[rl] = softmax_scale * (ds @ k)
        dk += softmax_scale * (ds.T @ q[rl])
        D[rl] = d_row
    return {"dq": dq, "dk": dk, "dv": dv, "D": D}


def attention_fwd_online(q, k, v, softmax_scale: float, causal: bool = False, tile_n: int = 128,
                         threshold: float = 8.0):
    """The conditional-rescale online softmax, in fp64, in the pages' order.

    Per query row, keys are visited in tiles of ``tile_n``. Scores are kept in
    log2 units, x_ij = scale * log2(e) * q_i . k_j. With m_tile the tile's row
    max and m_used the max currently used for exponentiation:
      * if m_tile > m_used + threshold (always true for the first visible tile):
        m_new = m_tile, and the running output and sum are multiplied by
        2^(m_used - m_new)  (a rescale);
      * otherwise the stale m_used is kept (the rescale is skipped), so every
        p_ij = 2^(x_ij - m_used) stays <= 2^threshold;
      * l += sum_j p_ij, acc += sum_j p_ij v_j.
    After the last tile the exact normalisation O = acc / l is applied, and
    LSE = ln(2) * (m_used + log2 l).

    Returns (O, LSE, stats) where stats counts rescales that happened and the
    rescale opportunities (visible tiles after a row's first visible tile).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    nq, nk, dv = q.shape[0], k.shape[0], v.shape[1]
    m_used = np.full(nq, -np.inf)
    l = np.zeros(nq)
    acc = np.zeros((nq, dv))
    seen = np.zeros(nq, dtype=bool)
    stats = {"rescales": 0, "opportunities": 0, "first_tiles": 0}
    if nq == 0 or nk == 0:
        return acc, np.full(nq, -np.inf), stats
    rows = np.arange(nq)
    lim = visible_limit(rows, nq, nk, causal)
    x_scale = softmax_scale * LOG2E
    for t0 in range(0, nk, tile_n):
        t1 = min(nk, t0 + tile_n)
        x = x_scale * (q @ k[t0:t1].T)
        cols = np.arange(t0, t1)
        x[cols[None, :] >= lim[:, None]] = -np.inf
        m_tile = x.max(axis=1)
        active = np.isfinite(m_tile)
        need = m_tile > m_used + threshold
        stats["first_tiles"] += int((active & ~seen).sum())
        stats["opportunities"] += int((active & seen).sum())
        stats["rescales"] += int((need & seen).sum())
        m_new = np.where(need, m_tile, m_used)
        alpha = np.where(need & seen, np.exp2(np.where(seen, m_used, 0.0) - m_new), 1.0)
        acc *= alpha[:, None]
        l *= alpha
        m_used = m_new
        seen |= active
        live = np.isfinite(m_used)
        p = np.zeros_like(x)
        p[live] = np.exp2(x[live] - m_used[live, None])
        l += p.sum(axis=1)
        acc += p @ v[t0:t1]
    o = np.zeros((nq, dv))
    lse = np.full(nq, -np.inf)
    ok = l > 0
    o[ok] = acc[ok] / l[ok, None]
    lse[ok] = LN2 * (m_used[ok] + np.log2(l[ok]))
    return o, lse, stats


def _seq_bounds(cu):
    cu = [int(x) for x in np.asarray(cu).reshape(-1)]
    return list(zip(cu[:-1], cu[1:]))


def head_score_mod(score_mod, h: int):
    """The score modification of head h: ALiBi takes a per-head slope list."""
    if score_mod is None or score_mod[0] != "alibi" or np.ndim(score_mod[1]) == 0:
        return score_mod
    return ("alibi", float(np.asarray(score_mod[1]).reshape(-1)[h]))


def attention_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, softmax_scale: float, causal: bool = False,
                         seqs=None, heads=None, row_block=None, score_mod=None):
    """Variable-length packed batch: q [total_q, H, d_qk], k/v [total_k, H, d].

    Each sequence s attends only within itself (rows cu_q[s]:cu_q[s+1] against
    keys cu_k[s]:cu_k[s+1]), each head independently. ``seqs`` / ``heads``
    select a subset (others are left as NaN). ``score_mod`` as in
    :func:`score_mod_apply`, positions counted within each sequence; ALiBi may
    give one slope per head. Returns (O [total_q, H, d_v], LSE [H, total_q]).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    tq, H = q.shape[0], q.shape[1]
    o = np.full((tq, H, v.shape[2]), np.nan)
    lse = np.full((H, tq), np.nan)
    bq, bk = _seq_bounds(cu_seqlens_q), _seq_bounds(cu_seqlens_k)
    for s in (range(len(bq)) if seqs is None else seqs):
        (q0, q1), (k0, k1) = bq[s], bk[s]
        for h in (range(H) if heads is None else heads):
            oo, ll = attention_fwd(q[q0:q1, h], k[k0:k1, h], v[k0:k1, h], softmax_scale, causal, row_block,
                                   score_mod=head_score_mod(score_mod, h))
            o[q0:q1, h] = oo
            lse[h, q0:q1] = ll
    return o, lse


def attention_bwd_varlen(q, k, v, do, cu_seqlens_q, cu_seqlens_k, softmax_scale: float, causal: bool = False,
                         seqs=None, heads=None, row_block=None, score_mod=None):
    """Backward of :func:`attention_fwd_varlen`; returns (dq, dk, dv) packed (NaN outside the subset)."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    dq = np.full(q.shape, np.nan)
    dk = np.full(k.shape, np.nan)
    dv = np.full(v.shape, np.nan)
    H = q.shape[1]
    bq, bk = _seq_bounds(cu_seqlens_q), _seq_bounds(cu_seqlens_k)
    for s in (range(len(bq)) if seqs is None else seqs):
        (q0, q1), (k0, k1) = bq[s], bk[s]
        for h in (range(H) if heads is None else heads):
            g = attention_bwd(q[q0:q1, h], k[k0:k1, h], v[k0:k1, h], do[q0:q1, h], softmax_scale, causal,
                              row_block, score_mod=head_score_mod(score_mod, h))
            dq[q0:q1, h] = g["dq"]
            dk[k0:k1, h] = g["dk"]
            dv[k0:k1, h] = g["dv"]
    return dq, dk, dv
