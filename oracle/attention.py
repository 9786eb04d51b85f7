"""fp64 decode attention through a block table -- the plain definition.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

What is computed (PagedAttention pages):
  * One query token per (sequence, query head) attends over that sequence's
    whole cached history -- decode phase, "AI Inference Serving at Scale",
    section 1; thewebvale section 1 (attend to all preceding tokens).
  * Token t of a sequence lives in physical block ``block_table[t // B]`` at
    offset ``t % B`` -- thewebvale section 2, "The Block Table" formula.
  * The result is the same as ordinary un-paged attention -- ontq section 8
    FAQ ("Does PagedAttention alter the mathematical accuracy ...").
  * Grouped-query attention: one KV head serves a group of query heads --
    ontq section 6.  Reading taken: query head h uses KV head h // g with
    g = Hq / Hkv (consecutive groups).

Softmax attention itself is textbook: s_t = scale * <q, k_t>,
p_t = exp(s_t - max_u s_u) / sum_u exp(s_u - max_u s_u), out = sum_t p_t v_t.
The scale is the caller's fp32 value widened to fp64.  A sequence with no
tokens yields a zero row.
"""

from __future__ import annotations

import numpy as np


def f64(x) -> np.ndarray:
    """Widen a torch tensor or array to fp64 numpy (exact for fp16 / bf16)."""
    if hasattr(x, "detach"):
        return x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)


def _i64(x) -> np.ndarray:
    if hasattr(x, "detach"):
        return x.detach().to("cpu").numpy().astype(np.int64)
    return np.asarray(x, dtype=np.int64)


def physical_location(block_table_row, t: int, block_size: int):
    """Token position t -> (physical block id, offset within the block)."""
    i = t // block_size           # logical block index
    j = t % block_size            # offset inside the block
    return int(block_table_row[i]), j


def _fetch_blocks(pool, ids, kv_head):
    """Copy the listed blocks of one KV head to host fp64: {block id: [B, d]}.
    Works for host or device tensors; only the listed blocks leave the pool."""
    uniq = sorted(set(int(i) for i in ids))
    if hasattr(pool, "detach"):
        import torch
        idx = torch.tensor(uniq, dtype=torch.long, device=pool.device)
        rows = pool.index_select(0, idx)[:, kv_head].to("cpu").double().numpy()
    else:
        rows = np.asarray(pool, dtype=np.float64)[uniq, kv_head]
    return {bid: rows[n] for n, bid in enumerate(uniq)}


def gather_sequence(k_pool, v_pool, block_table_row, ctx: int, kv_head: int, block_size: int):
    """Walk the block table token by token and collect K, V rows [ctx, d] (fp64)."""
    nblk = -(-ctx // block_size)
    ids = [int(block_table_row[i]) for i in range(nblk)]
    kb = _fetch_blocks(k_pool, ids, kv_head)
    vb = _fetch_blocks(v_pool, ids, kv_head)
    d = k_pool.shape[-1]
    K = np.empty((ctx, d))
    V = np.empty((ctx, d))
    for t in range(ctx):
        blk, off = physical_location(block_table_row, t, block_size)
        K[t] = kb[blk][off]
        V[t] = vb[blk][off]
    return K, V


def softmax_weights(q_row: np.ndarray, K: np.ndarray, scale: float) -> np.ndarray:
    """p_t for one query row over keys K [ctx, d]."""
    s = scale * (K @ q_row)
    e = np.exp(s - s.max())
    return e / e.sum()


def decode_ref(q, k_pool, v_pool, block_tables, context_lens, scale: float,
               rows=None) -> np.ndarray:
    """Paged decode attention in fp64.

    q [N, Hq, d]; k_pool, v_pool [NB, Hkv, B, d] (host or device tensors, or
    arrays); block_tables [N, MB]; context_lens [N].  Returns out [N, Hq, d]
    in fp64.  ``rows`` restricts the work to a list of (seq, q_head) pairs;
    the other rows are left NaN.
    """
    qf = f64(q)
    bt = _i64(block_tables)
    cl = _i64(context_lens)
    N, Hq, d = qf.shape
    Hkv, B = k_pool.shape[1], k_pool.shape[2]
    g = Hq // Hkv
    out = np.full((N, Hq, d), np.nan)
    todo = [(b, h) for b in range(N) for h in range(Hq)] if rows is None else list(rows)
    cache = {}
    for b, h in todo:
        ctx = int(cl[b])
        if ctx == 0:
            out[b, h] = 0.0
            continue
        kh = h // g
        if (b, kh) not in cache:
            cache = {(b, kh): gather_sequence(k_pool, v_pool, bt[b], ctx, kh, B)}
        K, V = cache[(b, kh)]
        p = softmax_weights(qf[b, h], K, scale)
        out[b, h] = p @ V
    return out


def unpaged_ref(q_seq, k_seq, v_seq, scale: float) -> np.ndarray:
    """Textbook attention over a contiguous cache -- the pre-paging layout.

    q_seq [Hq, d]; k_seq, v_seq [ctx, Hkv, d] contiguous.  Dense matrix form:
    S = scale * Q K^T per KV head group, row softmax, O = P V.
    """
    qf, kf, vf = f64(q_seq), f64(k_seq), f64(v_seq)
    Hq = qf.shape[0]
    Hkv = kf.shape[1]
    g = Hq // Hkv
    out = np.zeros_like(qf)
    if kf.shape[0] == 0:
        return out
    for kh in range(Hkv):
        Q = qf[kh * g:(kh + 1) * g]                 # [g, d]
        S = scale * Q @ kf[:, kh, :].T              # [g, ctx]
        S -= S.max(axis=1, keepdims=True)
        P = np.exp(S)
        P /= P.sum(axis=1, keepdims=True)
        out[kh * g:(kh + 1) * g] = P @ vf[:, kh, :]
    return out


# ---------------------------------------------------------------------------
# Partitioned form: split the keys into ranges, then merge with log-sum-exp.
# ---------------------------------------------------------------------------

def partial_ref(q_row, K, V, scale: float, lo: int, hi: int):
    """Attention state of keys [lo, hi): (m, l, o) with m = max score,
    l = sum exp(s - m), o = sum exp(s - m) v (not normalised)."""
    s = scale * (K[lo:hi] @ q_row)
    m = s.max()
    e = np.exp(s - m)
    return m, e.sum(), e @ V[lo:hi]


def lse_merge_ref(parts) -> np.ndarray:
    """Combine partition states: M = max m_p, L = sum l_p e^{m_p - M},
    out = sum o_p e^{m_p - M} / L."""
    M = max(m for m, _, _ in parts)
    L = sum(l * np.exp(m - M) for m, l, _ in parts)
    O = sum(o * np.exp(m - M) for m, _, o in parts)
    return O / L


# ---------------------------------------------------------------------------
# Shared prompt prefixes: sequences of a group point at the same leading
# blocks (ontq section 3, copy-on-write sharing of prompt blocks;
# letsbuildsolutions "Production Considerations", prefix caching).
# ---------------------------------------------------------------------------

def check_prefix_groups(block_tables, context_lens, group_starts, group_prefix_blocks, block_size):
    """True when every member of each group has the group's shared leading
    table entries and at least that many full blocks of context."""
    bt = _i64(block_tables)
    cl = _i64(context_lens)
    gs = [int(x) for x in group_starts]
    for gi, pblk in enumerate(int(x) for x in group_prefix_blocks):
        for s in range(gs[gi], gs[gi + 1]):
            if cl[s] < pblk * block_size:
                return False
            if any(bt[s, i] != bt[gs[gi], i] for i in range(pblk)):
                return False
    return True


def decode_shared_prefix_ref(q, k_pool, v_pool, block_tables, context_lens, scale, group_starts,
                             group_prefix_blocks, rows=None) -> np.ndarray:
    """Decode attention computed in two parts per row, as a prefix-aware
    kernel would: the shared prefix keys (read through the group's first
    member's table) and the row's own remaining keys, each reduced to a
    partition state and combined by the log-sum-exp rule.  Equal to
    ``decode_ref`` whenever the groups are consistent."""
    qf = f64(q)
    bt = _i64(block_tables)
    cl = _i64(context_lens)
    N, Hq, d = qf.shape
    Hkv, B = k_pool.shape[1], k_pool.shape[2]
    g = Hq // Hkv
    prefix_of = np.zeros(N, dtype=np.int64)
    owner = np.arange(N)
    gs = [int(x) for x in group_starts]
    for gi, pblk in enumerate(int(x) for x in group_prefix_blocks):
        for s in range(gs[gi], gs[gi + 1]):
            prefix_of[s] = pblk
            owner[s] = gs[gi]
    out = np.full((N, Hq, d), np.nan)
    todo = [(b, h) for b in range(N) for h in range(Hq)] if rows is None else list(rows)
    cache = {}
    for b, h in todo:
        ctx = int(cl[b])
        if ctx == 0:
            out[b, h] = 0.0
            continue
        kh = h // g
        npre = int(prefix_of[b]) * B
        if (b, kh) not in cache:
            K, V = gather_sequence(k_pool, v_pool, bt[b], ctx, kh, B)
            if npre:
                Kp, Vp = gather_sequence(k_pool, v_pool, bt[owner[b]], npre, kh, B)
                K = np.concatenate([Kp, K[npre:]])
                V = np.concatenate([Vp, V[npre:]])
            cache = {(b, kh): (K, V)}
        K, V = cache[(b, kh)]
        parts = [partial_ref(qf[b, h], K, V, scale, lo, hi)
                 for lo, hi in ((0, npre), (npre, ctx)) if hi > lo]
        out[b, h] = lse_merge_ref(parts)
    return out


# ---------------------------------------------------------------------------
# Multi-token query: a chunk of new tokens per sequence, causal within it.
# ---------------------------------------------------------------------------

def decode_multi_ref(q, k_pool, v_pool, block_tables, context_lens, q_start, scale: float) -> np.ndarray:
    """Paged attention for a chunk of query tokens per sequence, in fp64.

    The pages' chunked prefill (thewebvale section 4: a long prompt is fed in
    chunks co-scheduled with decode) and speculative verification
    (letsbuildsolutions "Speculative Decoding", ontq section 7: the target
    model scores all drafted tokens in one pass) both need attention for
    several new tokens of one sequence at once.  Reading taken: sequence b's
    q_len = q_start[b + 1] - q_start[b] query tokens are its last q_len cached
    tokens (their K/V were appended before the call), at positions
    ctx - q_len .. ctx - 1, and query token i attends causally to keys
    t <= ctx - q_len + i.  q [T, Hq, d] with T = q_start[N], sequence b's
    rows at q_start[b] ..; returns out [T, Hq, d].
    """
    qf = f64(q)
    bt = _i64(block_tables)
    cl = _i64(context_lens)
    qs = _i64(q_start)
    T, Hq, d = qf.shape
    Hkv, B = k_pool.shape[1], k_pool.shape[2]
    g = Hq // Hkv
    out = np.full((T, Hq, d), np.nan)
    for b in range(len(cl)):
        ctx, r0, r1 = int(cl[b]), int(qs[b]), int(qs[b + 1])
        n = r1 - r0
        assert 0 <= n <= ctx or (n == 0 and ctx == 0), "a chunk longer than its context"
        for kh in range(Hkv):
            if n == 0:
                continue
            K, V = gather_sequence(k_pool, v_pool, bt[b], ctx, kh, B)
            for i in range(n):
                lim = ctx - n + i                          # last key this token sees
                for h in range(kh * g, (kh + 1) * g):
                    p = softmax_weights(qf[r0 + i, h], K[:lim + 1], scale)
                    out[r0 + i, h] = p @ V[:lim + 1]
    return out


def causal_dense_ref(q_all, k_seq, v_seq, scale: float) -> np.ndarray:
    """Textbook causal self-attention over one contiguous sequence:
    q_all [ctx, Hq, d], k_seq, v_seq [ctx, Hkv, d]; S = scale Q K^T with
    S[i, t] = -inf for t > i, row softmax, O = P V.  Returns [ctx, Hq, d]."""
    qf, kf, vf = f64(q_all), f64(k_seq), f64(v_seq)
    ctx, Hq, d = qf.shape
    Hkv = kf.shape[1]
    g = Hq // Hkv
    out = np.zeros_like(qf)
    mask = np.triu(np.ones((ctx, ctx), dtype=bool), k=1)
    for h in range(Hq):
        kh = h // g
        S = scale * qf[:, h, :] @ kf[:, kh, :].T
        S[mask] = -np.inf
        S -= S.max(axis=1, keepdims=True)
        P = np.exp(S)
        P /= P.sum(axis=1, keepdims=True)
        out[:, h, :] = P @ vf[:, kh, :]
    return out
