"""Plain fp64 restatement of context-parallel causal ring attention.

TEST INFRASTRUCTURE ONLY (see the package docstring): no product code may
import this module.

Sources (page title, then section):
* [MaxText] "Announcing Long-Context Training on TPUs with MaxText Context
  Parallelism": "Context Parallelism in MaxText" (P2P ring attention: KV
  chunks move one hop per step, each chip attends its queries to the chunk it
  holds and merges partial results as it goes) and "Built on a fast attention
  kernel" (block-sparse flash attention that skips fully masked blocks and
  handles packed sequences; called once per ring step, forward and
  backward).
* [CP-Inference] "Context Parallelism for Scalable Million-Token Inference":
  "Attention Compute Patterns in Multi-Turn Chat" (full prefill is the lower
  triangle; partial prefill lets new tokens see the cached prefix and their
  own triangle), "Load Balancing in CP" (2R chunks, two per rank, worked
  example with 4 tokens and 2 ranks), "Ring Attention Algorithms" (Pass KV:
  Q stays, KV circulates, partial outputs merged at the end; Pass Q: KV
  stays, Q circulates, partial outputs permuted back to order, returned to
  their owners by an all-to-all, then merged), and "Context Parallelism (CP)
  vs. Tensor Parallelism (TP)" (grouped-query heads: few KV heads shared by
  many Q heads).

Readings where the pages are silent:
* Rank r holds chunks r and 2R-1-r, in that order ("Load Balancing in CP"
  says rank 0 may take the first and last chunk).
* Ring direction: at step t rank r holds the KV (Pass KV) or the Q (Pass Q)
  that rank (r - t) mod R started with.
* The merge is the log-sum-exp combination of partial softmax results
  (the pages name the "merge attention operation" but print no formula):
  LSE = M + ln sum_i exp(LSE_i - M), O = sum_i exp(LSE_i - LSE) O_i.
* LSE is natural-log, with the softmax scale applied to the scores.
* A row that sees no key in a step has O = 0 and LSE = -inf there.
* GQA: query head h uses KV head h // G (contiguous groups).
* Packed sequences: a key is visible iff it lies in the same document as the
  query and at a position not after it. Documents are given by cu_seqlens
  in natural token positions.
* Partial prefill: cache and new tokens are each split 2R ways the same way;
  rank r's KV is [its cache chunks, its new chunks]; new token i sits at
  global position P + i (P = cached length).
* Backward: the standard softmax gradient with the global (merged) LSE, so
  each ring step's share uses P = exp(S - LSE_global).
* Sliding window ([MaxText] "What's next": models that mix sliding-window
  and global layers): with a window of W tokens a key is visible only if
  it is also fewer than W positions behind the query (q - k < W); W = 0
  means no window.
* Pass KV or Pass Q ([CP-Inference] "Ring Attention Algorithms" and "Context
  Parallelism (CP) vs. Tensor Parallelism (TP)"): the ring message of Pass Q
  is the new tokens' Q (T_new * Hq * d), that of Pass KV the K and V of all
  tokens (2 * T_total * Hkv * d); the cheaper one is chosen (Pass Q only
  when strictly smaller).
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "rank_chunks",
    "shard_positions",
    "plan_positions",
    "batch_cu_seqlens",
    "ring_schedule",
    "doc_index",
    "visible_mask",
    "block_mask",
    "work_list",
    "count_visible",
    "partial_attention",
    "attention",
    "lse_merge",
    "round_bf16",
    "ring_forward",
    "attention_backward",
    "ring_backward",
    "sampled_forward",
    "sampled_dq",
    "sampled_dkdv",
    "select_variant",
    "head_split",
    "head_gather",
    "decode",
    "TILE",
]

TILE = 128
EMPTY, PARTIAL, FULL = 0, 1, 2


# ---------------------------------------------------------------------------
# Chunk plan  ([CP-Inference] "Load Balancing in CP")
# ---------------------------------------------------------------------------
def rank_chunks(R: int, layout: str = "zigzag", a2a: int = 1):
    """Chunk indices held by each rank, in the rank's local order.

    zigzag: the sequence is cut into 2R chunks and rank r takes chunks r and
    2R-1-r. contiguous: R chunks, rank r takes chunk r (no balancing).
    usp ([MaxText] "A2A + P2P (USP)"): D = a2a * R devices, each holding its
    zigzag pair of 2D chunks; an all-to-all within each group of a2a
    consecutive devices pools the group's tokens, so ring rank r holds the
    chunks of devices r*a2a, ..., r*a2a + a2a - 1. The receiving devices may
    place the pooled chunks in any order; they are kept in ascending
    position order, so every rank's positions increase along its rows.
    """
    if layout == "zigzag":
        return [[r, 2 * R - 1 - r] for r in range(R)]
    if layout == "contiguous":
        return [[r] for r in range(R)]
    if layout == "usp":
        D = a2a * R
        return [sorted(c for d in range(r * a2a, (r + 1) * a2a) for c in (d, 2 * D - 1 - d))
                for r in range(R)]
    raise ValueError(layout)


def shard_positions(n_tokens: int, R: int, layout: str = "zigzag",
                    offset: int = 0, a2a: int = 1):
    """Global positions held by each rank, in local order, for a run of
    ``n_tokens`` tokens starting at global position ``offset``."""
    chunks = rank_chunks(R, layout, a2a)
    n_chunks = {"zigzag": 2 * R, "contiguous": R, "usp": 2 * R * a2a}[layout]
    assert n_tokens % n_chunks == 0
    c = n_tokens // n_chunks
    out = []
    for r in range(R):
        pos = [np.arange(ch * c, (ch + 1) * c, dtype=np.int64) + offset
               for ch in chunks[r]]
        out.append(np.concatenate(pos))
    return out


def plan_positions(seq_len: int, R: int, layout: str = "zigzag",
                   kv_prefix_len: int = 0, a2a: int = 1, batch: int = 1):
    """Per-rank global positions of the query tokens and of the KV tokens.

    Full prefill: Q and KV are the same tokens. Partial prefill (a cached
    prefix of length P): the cache and the new tokens are each sharded the
    same way; rank r's KV is its cache shard followed by its new-token shard,
    and the new tokens (the queries) sit at positions P, P+1, ...
    A batch of B independent sequences (reading: each one sharded on its
    own, a rank holding its part of sequence 0, then of sequence 1, ...)
    lives in one position space where sequence b starts at b*(P + seq_len);
    its documents must separate the sequences (batch_cu_seqlens).
    """
    P = int(kv_prefix_len)
    L = P + int(seq_len)
    q_pos = [[] for _ in range(R)]
    kv_pos = [[] for _ in range(R)]
    for b in range(int(batch)):
        new = shard_positions(seq_len, R, layout, offset=b * L + P, a2a=a2a)
        cache = shard_positions(P, R, layout, offset=b * L, a2a=a2a) if P else None
        for r in range(R):
            q_pos[r].append(new[r])
            if cache is not None:
                kv_pos[r].append(cache[r])
            kv_pos[r].append(new[r])
    q_pos = [np.concatenate(x) for x in q_pos]
    kv_pos = [np.concatenate(x) for x in kv_pos]
    return q_pos, kv_pos


def batch_cu_seqlens(seq_len: int, batch: int, kv_prefix_len: int = 0) -> np.ndarray:
    """Document offsets of a batch: one document per sequence of
    kv_prefix_len + seq_len positions."""
    L = int(kv_prefix_len) + int(seq_len)
    return np.arange(int(batch) + 1, dtype=np.int64) * L


def ring_schedule(R: int, variant: str = "pass_kv"):
    """sched[t][r] = (q_owner, kv_owner) of the pair rank r computes at step t.

    Pass KV: rank r keeps its Q and holds the KV that started on rank
    (r - t) mod R. Pass Q: rank r keeps its KV and holds the Q that started
    on rank (r - t) mod R.
    """
    sched = []
    for t in range(R):
        row = []
        for r in range(R):
            other = (r - t) % R
            if variant == "pass_kv":
                row.append((r, other))
            elif variant == "pass_q":
                row.append((other, r))
            else:
                raise ValueError(variant)
        sched.append(row)
    return sched


# ---------------------------------------------------------------------------
# Mask  ([CP-Inference] "Attention Compute Patterns in Multi-Turn Chat";
#        [MaxText] "Built on a fast attention kernel": packed sequences)
# ---------------------------------------------------------------------------
def doc_index(pos: np.ndarray, cu_seqlens) -> np.ndarray:
    """Document id of each global position (all zero without documents)."""
    pos = np.asarray(pos, dtype=np.int64)
    if cu_seqlens is None:
        return np.zeros(pos.shape, dtype=np.int64)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    return np.searchsorted(cu, pos, side="right") - 1


def _vis(qp, qd, kp, kd, window):
    """Visibility of keys (kp, kd) from queries (qp, qd): same document, not
    after the query, and (with a window) fewer than `window` positions
    behind it."""
    v = (kp[None, :] <= qp[:, None]) & (kd[None, :] == qd[:, None])
    if window:
        v &= (qp[:, None] - kp[None, :]) < window
    return v


def visible_mask(qpos, kpos, cu_seqlens=None, *, window: int = 0) -> np.ndarray:
    """vis[i, j]: key at kpos[j] is visible from the query at qpos[i]."""
    qpos = np.asarray(qpos, dtype=np.int64)
    kpos = np.asarray(kpos, dtype=np.int64)
    return _vis(qpos, doc_index(qpos, cu_seqlens), kpos, doc_index(kpos, cu_seqlens),
                window)


def block_mask(q_pos, kv_pos, cu_seqlens=None, tile: int = TILE, *, window: int = 0):
    """Tile class per (q_owner, kv_owner, q_tile, kv_tile), by brute force.

    EMPTY (0) if no (query, key) pair of the tile is visible, FULL (2) if all
    are, PARTIAL (1) otherwise. Computed from the elementwise mask with
    ``any``/``all`` over each tile.
    """
    R = len(q_pos)
    nq = len(q_pos[0])
    nk = len(kv_pos[0])
    assert nq % tile == 0 and nk % tile == 0
    out = np.zeros((R, R, nq // tile, nk // tile), dtype=np.uint8)
    for a in range(R):
        for b in range(R):
            vis = visible_mask(q_pos[a], kv_pos[b], cu_seqlens, window=window)
            v4 = vis.reshape(nq // tile, tile, nk // tile, tile)
            anyv = v4.any(axis=(1, 3))
            allv = v4.all(axis=(1, 3))
            out[a, b] = np.where(allv, FULL, np.where(anyv, PARTIAL, EMPTY))
    return out


def work_list(bm, sched, step: int, backward: bool = False) -> np.ndarray:
    """The compacted work list of ring step ``step`` from the block classes
    bm[q_owner][kv_owner][q tile][kv tile] ([MaxText] "Built on a fast
    attention kernel": fully masked blocks are skipped). Reading: the step's
    pairs are taken in rank order and their tiles in order; forward, one
    item per query tile with the run [lo, hi) of its non-empty key tiles
    (lo = hi = 0 when there is none); backward, one item per key tile that
    has a non-empty run of query tiles. A run must be contiguous. The list is
    then sorted by run length, longest first, equal lengths keeping their
    order. Rows: q_owner, kv_owner, tile, lo, hi, number of FULL tiles."""
    items = []
    for qo, ko in sched[step]:
        m = np.asarray(bm[qo][ko])
        n_tiles = m.shape[1] if backward else m.shape[0]
        for t in range(n_tiles):
            line = m[:, t] if backward else m[t]
            nz = np.nonzero(line)[0]
            if len(nz) == 0:
                if not backward:
                    items.append((qo, ko, t, 0, 0, 0))
                continue
            lo, hi = int(nz[0]), int(nz[-1]) + 1
            assert len(nz) == hi - lo, "non-contiguous run of visible tiles"
            items.append((qo, ko, t, lo, hi, int((line[lo:hi] == FULL).sum())))
    items.sort(key=lambda it: -(it[4] - it[3]))   # list.sort is stable
    return np.array(items, dtype=np.int64).reshape(-1, 6)


def count_visible(qpos, kpos, cu_seqlens=None, *, window: int = 0) -> int:
    """Number of visible (query, key) pairs (per query head)."""
    return int(visible_mask(qpos, kpos, cu_seqlens, window=window).sum())


# ---------------------------------------------------------------------------
# Attention and merge
# ---------------------------------------------------------------------------
def _as_f64(x):
    return np.asarray(x, dtype=np.float64)


def _key_index(keep):
    """Indices of kept keys; a slice when they are one contiguous run."""
    kidx = np.nonzero(keep)[0]
    if kidx.size and kidx[-1] - kidx[0] + 1 == kidx.size:
        return slice(int(kidx[0]), int(kidx[-1]) + 1), kidx
    return kidx, kidx


def _per_head(x):
    """[m, H, d] -> list of H contiguous [m, d] fp64 arrays."""
    return [np.ascontiguousarray(x[:, h, :], dtype=np.float64)
            for h in range(x.shape[1])]


def partial_attention(q, k, v, qpos, kpos, cu_seqlens=None, scale=None,
                      row_block: int = 512, *, window: int = 0):
    """Softmax attention of queries ``q`` over keys ``k``/values ``v``.

    q: [n, Hq, d], k and v: [m, Hkv, d]. Returns O [n, Hq, d] and LSE [Hq, n]
    (natural log of the sum of exp(scale * q.k) over the visible keys), in
    fp64. Each row's softmax is taken over that row's complete visible set in
    two passes (max, then exp and sum). Rows with no visible key get O = 0
    and LSE = -inf. Rows are processed in blocks only to bound memory; keys
    outside every row's [document start, position] range of a block are
    skipped because they are invisible to all of its rows.
    """
    q = _as_f64(q)
    n, Hq, d = q.shape
    m, Hkv, _ = k.shape
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    kh_ = _per_head(k)
    vh_ = _per_head(v)
    qpos = np.asarray(qpos, dtype=np.int64)
    kpos = np.asarray(kpos, dtype=np.int64)
    qdoc = doc_index(qpos, cu_seqlens)
    kdoc = doc_index(kpos, cu_seqlens)
    O = np.zeros((n, Hq, d))
    LSE = np.full((Hq, n), -np.inf)
    for r0 in range(0, n, row_block):
        r1 = min(n, r0 + row_block)
        qp = qpos[r0:r1]
        qd = qdoc[r0:r1]
        keep = (kpos <= qp.max()) & (kdoc >= qd.min()) & (kdoc <= qd.max())
        if window:
            keep &= kpos > qp.min() - window
        ksel, kidx = _key_index(keep)
        if kidx.size == 0:
            continue
        vis = _vis(qp, qd, kpos[kidx], kdoc[kidx], window)
        has = vis.any(axis=1)
        for h in range(Hq):
            kh = h // G
            s = scale * (q[r0:r1, h, :] @ kh_[kh][ksel].T)
            s = np.where(vis, s, -np.inf)
            mx = s.max(axis=1)
            mx_safe = np.where(has, mx, 0.0)
            p = np.exp(s - mx_safe[:, None])
            l = p.sum(axis=1)
            l_safe = np.where(has, l, 1.0)
            o = (p @ vh_[kh][ksel]) / l_safe[:, None]
            O[r0:r1, h, :] = np.where(has[:, None], o, 0.0)
            LSE[h, r0:r1] = np.where(has, mx_safe + np.log(l_safe), -np.inf)
    return O, LSE


def attention(q, k, v, qpos, kpos, cu_seqlens=None, scale=None, *, window: int = 0):
    """Monolithic (no context parallelism) causal attention over all keys."""
    return partial_attention(q, k, v, qpos, kpos, cu_seqlens, scale, window=window)


def lse_merge(parts):
    """Merge partial results [(O_i [n,H,d], LSE_i [H,n]), ...] of disjoint
    key sets into the softmax result over their union."""
    lses = np.stack([_as_f64(p[1]) for p in parts])          # [k, H, n]
    outs = np.stack([_as_f64(p[0]) for p in parts])          # [k, n, H, d]
    M = lses.max(axis=0)                                     # [H, n]
    finite = np.isfinite(M)
    M_safe = np.where(finite, M, 0.0)
    w = np.exp(lses - M_safe[None])                          # 0 for -inf
    S = w.sum(axis=0)
    LSE = np.where(finite, M_safe + np.log(np.where(finite, S, 1.0)), -np.inf)
    LSE_safe = np.where(finite, LSE, 0.0)
    coef = np.where(finite[None], np.exp(lses - LSE_safe[None]), 0.0)  # [k,H,n]
    O = np.einsum("khn,knhd->nhd", coef, outs)
    return O, LSE


def _split(x, R):
    n = x.shape[0] // R
    return [x[r * n:(r + 1) * n] for r in range(R)]


def round_bf16(x):
    """Nearest bf16 value of each float64, ties to the even significand: 8
    significant bits over the fp32 exponent range; below 2^-126 the spacing
    stays 2^-133 (subnormals); magnitudes at or above the overflow point
    (2 - 2^-8) * 2^127 become infinite; NaN stays NaN. The storage rounding
    of bf16 partial outputs (reading: a plan with bf16 partials stores each
    ring step's O in this format before the merge)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    finite = np.isfinite(a)
    a0 = np.where(finite, a, 0.0)
    _, e = np.frexp(a0)                   # a = f * 2^e with f in [0.5, 1)
    e = np.maximum(e, -125)               # subnormals keep the spacing of 2^-126
    spacing = np.ldexp(1.0, e - 8)
    r = np.rint(a0 / spacing) * spacing   # a / spacing is exact; rint: half to even
    r = np.where(r >= 2.0 ** 128, np.inf, r)
    r = np.where(finite, r, a)
    return np.copysign(r, x)


def ring_forward(q, k, v, q_pos, kv_pos, cu_seqlens=None, scale=None,
                 variant: str = "pass_kv", *, window: int = 0, partial_dtype: str = "f32"):
    """Explicit ring over R virtual ranks; inputs in rank-major order.

    q: [R*n_q, Hq, d] (rank r's queries are rows r*n_q ...), k/v:
    [R*n_kv, Hkv, d]. Pass KV merges each step's partial result into a
    running result in step order. Pass Q stores the partial result of
    (q_owner, kv_owner) at the kv_owner's slot (the permutation back to
    order), hands each q_owner its R partials (the all-to-all), and merges
    them in kv_owner order; with partial_dtype "bf16" a slot holds its O
    rounded to bf16 (round_bf16; the LSE stays exact). Returns
    O [R*n_q, Hq, d], LSE [Hq, R*n_q].
    """
    if partial_dtype not in ("f32", "bf16"):
        raise ValueError("partial_dtype must be 'f32' or 'bf16'")
    R = len(q_pos)
    Q = _split(_as_f64(q), R)
    K = _split(_as_f64(k), R)
    V = _split(_as_f64(v), R)
    sched = ring_schedule(R, variant)
    if variant == "pass_kv":
        acc = [None] * R
        for t in range(R):
            for r in range(R):
                qo, ko = sched[t][r]
                part = partial_attention(Q[qo], K[ko], V[ko], q_pos[qo],
                                         kv_pos[ko], cu_seqlens, scale, window=window)
                acc[qo] = part if acc[qo] is None else lse_merge([acc[qo], part])
        outs = acc
    else:
        slots = [[None] * R for _ in range(R)]   # slots[q_owner][kv_owner]
        for t in range(R):
            for r in range(R):
                qo, ko = sched[t][r]
                o_t, l_t = partial_attention(Q[qo], K[ko], V[ko], q_pos[qo], kv_pos[ko],
                                             cu_seqlens, scale, window=window)
                slots[qo][ko] = (round_bf16(o_t) if partial_dtype == "bf16" else o_t, l_t)
        outs = [lse_merge(slots[qo]) for qo in range(R)]
    O = np.concatenate([o for o, _ in outs], axis=0)
    LSE = np.concatenate([l for _, l in outs], axis=1)
    return O, LSE


# ---------------------------------------------------------------------------
# Backward  (softmax gradient with recomputed probabilities)
# ---------------------------------------------------------------------------
def _pair_backward(q, k, v, dout, o, lse, qpos, kpos, cu_seqlens, scale,
                   dq, dk, dv, row_block: int = 512, want_dkdv: bool = True,
                   window: int = 0):
    """Add one (query set, key set) share of the gradients into dq/dk/dv.

    P = exp(scale q.k - LSE) on visible pairs (LSE = the merged, global one),
    dV += P^T dO, dP = dO V^T, D = rowsum(dO * O), dS = P (dP - D),
    dQ += scale dS K, dK += scale dS^T Q; dK and dV sum over the query heads
    of each KV head's group.
    """
    n, Hq, d = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    kh_ = _per_head(k)
    vh_ = _per_head(v)
    qpos = np.asarray(qpos, dtype=np.int64)
    kpos = np.asarray(kpos, dtype=np.int64)
    qdoc = doc_index(qpos, cu_seqlens)
    kdoc = doc_index(kpos, cu_seqlens)
    D = np.einsum("nhd,nhd->hn", dout, o)
    for r0 in range(0, n, row_block):
        r1 = min(n, r0 + row_block)
        qp = qpos[r0:r1]
        qd = qdoc[r0:r1]
        keep = (kpos <= qp.max()) & (kdoc >= qd.min()) & (kdoc <= qd.max())
        if window:
            keep &= kpos > qp.min() - window
        ksel, kidx = _key_index(keep)
        if kidx.size == 0:
            continue
        vis = _vis(qp, qd, kpos[kidx], kdoc[kidx], window)
        for h in range(Hq):
            kh = h // G
            kk = kh_[kh][ksel]
            s = scale * (q[r0:r1, h, :] @ kk.T)
            lse_h = lse[h, r0:r1]
            lse_safe = np.where(np.isfinite(lse_h), lse_h, 0.0)
            p = np.where(vis, np.exp(s - lse_safe[:, None]), 0.0)
            dp = dout[r0:r1, h, :] @ vh_[kh][ksel].T
            ds = p * (dp - D[h, r0:r1][:, None])
            dq[r0:r1, h, :] += scale * (ds @ kk)
            if want_dkdv:
                dv[ksel, kh, :] += p.T @ dout[r0:r1, h, :]
                dk[ksel, kh, :] += scale * (ds.T @ q[r0:r1, h, :])


def attention_backward(q, k, v, dout, o, lse, qpos, kpos, cu_seqlens=None,
                       scale=None, *, window: int = 0):
    """Gradients of monolithic attention. o/lse are the forward results."""
    q, k, v, dout, o, lse = map(_as_f64, (q, k, v, dout, o, lse))
    d = q.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    _pair_backward(q, k, v, dout, o, lse, qpos, kpos, cu_seqlens, scale,
                   dq, dk, dv, window=window)
    return dq, dk, dv


def ring_backward(q, k, v, dout, o, lse, q_pos, kv_pos, cu_seqlens=None,
                  scale=None, variant: str = "pass_kv", steps=None, *, window: int = 0):
    """Explicit ring backward: each step adds the share of the pair it holds.

    Rank-major inputs as in ``ring_forward``; o and lse are the merged
    forward results. dQ of a pair lands at its q_owner, dK/dV at its
    kv_owner (in a real ring they travel back with the chunk). ``steps``
    restricts the sum to those ring steps (default: all of them).
    """
    q, k, v, dout, o, lse = map(_as_f64, (q, k, v, dout, o, lse))
    R = len(q_pos)
    d = q.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    nq = q.shape[0] // R
    nk = k.shape[0] // R
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for t, row in enumerate(ring_schedule(R, variant)):
        if steps is not None and t not in steps:
            continue
        for qo, ko in row:
            qs = slice(qo * nq, (qo + 1) * nq)
            ks = slice(ko * nk, (ko + 1) * nk)
            dq_p = np.zeros((nq,) + q.shape[1:])
            dk_p = np.zeros((nk,) + k.shape[1:])
            dv_p = np.zeros((nk,) + v.shape[1:])
            _pair_backward(q[qs], k[ks], v[ks], dout[qs], o[qs], lse[:, qs],
                           q_pos[qo], kv_pos[ko], cu_seqlens, scale,
                           dq_p, dk_p, dv_p, window=window)
            dq[qs] += dq_p
            dk[ks] += dk_p
            dv[ks] += dv_p
    return dq, dk, dv


# ---------------------------------------------------------------------------
# Sampled rows for workloads too large for the full oracle
# ---------------------------------------------------------------------------
def sampled_forward(q, k, v, rows, qpos, kpos, cu_seqlens=None, scale=None,
                    row_block: int = 32, *, window: int = 0):
    """O [len(rows), Hq, d] and LSE [Hq, len(rows)] at the given query rows,
    each an exact full-prefix softmax over all of that row's visible keys."""
    rows = np.asarray(rows, dtype=np.int64)
    return partial_attention(_as_f64(np.asarray(q)[rows]), k, v,
                             np.asarray(qpos)[rows], kpos, cu_seqlens, scale,
                             row_block=row_block, window=window)


def sampled_dq(q, k, v, dout, rows, qpos, kpos, cu_seqlens=None, scale=None,
               row_block: int = 32, *, window: int = 0):
    """dQ at the given rows, using the oracle's own O and LSE of those rows."""
    d = q.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    rows = np.asarray(rows, dtype=np.int64)
    o, lse = sampled_forward(q, k, v, rows, qpos, kpos, cu_seqlens, scale,
                             row_block, window=window)
    q_rows = _as_f64(np.asarray(q)[rows])
    dout_rows = _as_f64(np.asarray(dout)[rows])
    dq = np.zeros_like(q_rows)
    _pair_backward(q_rows, k, v, dout_rows, o, lse,
                   np.asarray(qpos)[rows], kpos, cu_seqlens, scale,
                   dq, None, None, row_block=row_block, want_dkdv=False,
                   window=window)
    return dq


def sampled_dkdv(q, k, v, dout, key_rows, qpos, kpos, cu_seqlens=None,
                 scale=None, *, window: int = 0):
    """dK and dV at the given key rows.

    Only the queries that can see one of those keys contribute; for each of
    them the full-prefix O and LSE are computed first. Returns
    (dk [len(key_rows), Hkv, d], dv [...]).
    """
    q = np.asarray(q)
    d = q.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    qpos = np.asarray(qpos, dtype=np.int64)
    kpos = np.asarray(kpos, dtype=np.int64)
    key_rows = np.asarray(key_rows, dtype=np.int64)
    kp = kpos[key_rows]
    vis = visible_mask(qpos, kp, cu_seqlens, window=window)
    qrows = np.nonzero(vis.any(axis=1))[0]
    o, lse = sampled_forward(q, k, v, qrows, qpos, kpos, cu_seqlens, scale,
                             window=window)
    kk = _as_f64(np.asarray(k)[key_rows])
    vv = _as_f64(np.asarray(v)[key_rows])
    dq = np.zeros((len(qrows),) + q.shape[1:])
    dk = np.zeros_like(kk)
    dv = np.zeros_like(vv)
    _pair_backward(_as_f64(q[qrows]), kk, vv, _as_f64(np.asarray(dout)[qrows]),
                   o, lse, qpos[qrows], kp, cu_seqlens, scale, dq, dk, dv,
                   window=window)
    return dk, dv


# ---------------------------------------------------------------------------
# Ring ordering choice  ([CP-Inference] "Ring Attention Algorithms")
# ---------------------------------------------------------------------------
def select_variant(n_new: int, n_cached: int, n_q_heads: int, n_kv_heads: int) -> str:
    """"pass_q" when the per-hop message of Pass Q (the Q of the n_new new
    tokens: n_new * Hq * d elements) is strictly smaller than that of Pass KV
    (K and V of all n_new + n_cached tokens: 2 * (n_new + n_cached) * Hkv * d),
    else "pass_kv". The head dimension d is common to both and drops out."""
    q_msg = n_new * n_q_heads
    kv_msg = 2 * (n_new + n_cached) * n_kv_heads
    return "pass_q" if q_msg < kv_msg else "pass_kv"


# ---------------------------------------------------------------------------
# Sequence <-> head all-to-all  ([MaxText] "All-to-All (Ulysses)", "A2A + P2P")
# ---------------------------------------------------------------------------
def head_split(x, a2a: int):
    """The all-to-all before attention, seen from one GPU holding every
    device's buffer. x: [T, H, e] with rows in device order (each device's
    tokens, all heads). Device u of a group keeps heads [u*H/a2a, (u+1)*H/a2a)
    and receives the group's other tokens for them; gathered over all groups,
    sub-rank u's tensor is x[:, its heads, :]. Returns [a2a, T, H/a2a, e]."""
    x = np.asarray(x)
    T, H = x.shape[0], x.shape[1]
    assert H % a2a == 0
    hs = H // a2a
    return np.stack([x[:, u * hs:(u + 1) * hs] for u in range(a2a)])


def head_gather(y):
    """The all-to-all after attention: the inverse of head_split. y:
    [a2a, T, H/a2a, e] -> [T, H, e]."""
    y = np.asarray(y)
    return np.concatenate([y[u] for u in range(y.shape[0])], axis=1)


# ---------------------------------------------------------------------------
# Decode  ([CP-Inference] "Attention Compute Patterns in Multi-Turn Chat",
# "Ring Attention Algorithms": Pass Q for decode)
# ---------------------------------------------------------------------------
def decode(q, k, v, R: int, scale=None):
    """One new query row per sequence attending to all of its keys.

    q: [B, Hq, d]; k, v: [B, T, Hkv, d], where the new token is the last of
    the T keys, so every key is visible. Rank r holds keys
    [r*T/R, (r+1)*T/R) of each sequence; the row visits every rank, each rank
    computes its partial attention, and the partials are merged. Returns
    O [B, Hq, d] and LSE [Hq, B]."""
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    B, T = k.shape[0], k.shape[1]
    assert T % R == 0
    n = T // R
    O = np.zeros(q.shape)
    LSE = np.zeros((q.shape[1], B))
    for b in range(B):
        parts = [partial_attention(q[b:b + 1], k[b, r * n:(r + 1) * n], v[b, r * n:(r + 1) * n],
                                   [T - 1], np.arange(r * n, (r + 1) * n), None, scale)
                 for r in range(R)]
        o, l = lse_merge(parts)
        O[b] = o[0]
        LSE[:, b] = l[:, 0]
    return O, LSE
