"""Float64 CPU oracle for exact (softmax) attention, its gradient, and split-KV decoding.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA path and imports nothing from the product package.

Every function works in float64 on whatever values it is given (the tests pass
the bf16-rounded inputs widened to float64).  NumPy's ``matmul``, ``exp``,
``log`` and ``max`` are the only library primitives used; there is no blocking,
fusion or reordering beyond what the cited definition or algorithm states.

Sources (web pages on exact tiled attention; cited by title and section):

* "attention_kernels.py" (CMU 15-779, lecture 5): section 1 ``SoftmaxState`` /
  ``merge_states`` / ``state_of_scores``; section 2 ``_scale``, ``_mask`` and
  ``standard_attention``; section 3 ``flash_forward`` (the block-wise loop and
  its ``stats`` counters); section 4 ``flash_backward`` (its docstring derives
  dS = P * (dP - D) from the softmax Jacobian diag(p) - p p^T, and its
  "dq_atomic_adds" counter); section 5 ``flash_decode``; section 6
  ``io_flash``.
* "lab.py" (hs-black, flash-attention post): ``dense``, ``tiled`` (row-wise
  online softmax returning the log-sum-exp) and ``backward`` (row-wise tiled
  gradient).
* "flash_attention_numpy.py" (first_principles, flash-attention tier 1):
  ``standard_attention`` with *unscaled* scores (scale = 1), used by the
  worked N=3, d=2 example, and ``flash_attention_tier1`` (the first
  algorithm's key-major loop order).

Pins (what each function is checked against, in ``tests/test_oracle_*.py``):
the printed N=3, d=2 example and hand-derived closed forms of it, uniform
scores giving the mean of V, N=1 and first-causal-row special cases,
``scipy.special.logsumexp`` / ``softmax`` on the dense path, block-size
invariance of the row-wise tiled path against the dense path (uneven last
tiles included), finiteness at x100 logits, central finite differences and
float64 autograd for both gradient paths, gradient invariants, the
algebraic laws of ``merge_states`` (identity, commutativity, associativity)
with split decoding equal to dense attention for every split count, and for
the block-wise loop: equality with the dense path for even and uneven blocks,
its counters against closed forms and an element-wise brute force, and
``io_flash`` against hand-computed values.  No function here is "parity
unpinned".
"""
from __future__ import annotations

from dataclasses import dataclass
from fractions import Fraction

import numpy as np

NEG_INF = -np.inf

# Query rows handled per matmul by the dense paths.  Softmax attention is
# defined row by row, so splitting the query axis changes nothing but peak
# memory (one chunk of full score rows at a time).
_ROW_CHUNK = 1024


def default_scale(d: int, scale: float | None) -> float:
    """Score scale: 1/sqrt(d) unless given ("attention_kernels.py", section 2, ``_scale``)."""
    return 1.0 / np.sqrt(d) if scale is None else float(scale)


def causal_mask(q_start: int, nq: int, nk: int, k_start: int = 0) -> np.ndarray:
    """Boolean (nq, nk) mask, True where the key is in the future of the query.

    Query row i sits at absolute position q_start + i and key column j at
    k_start + j; the key is hidden when its position exceeds the query's
    ("attention_kernels.py", section 2, ``_mask``).
    """
    qpos = np.arange(q_start, q_start + nq)[:, None]
    kpos = np.arange(k_start, k_start + nk)[None, :]
    return kpos > qpos


def _as_f64(*arrays):
    return [np.asarray(a, dtype=np.float64) for a in arrays]


def _heads(x: np.ndarray):
    """Iterate over the leading (batch, head, ...) indices of a (..., N, d) array."""
    return np.ndindex(*x.shape[:-2])


# --------------------------------------------------------------------------
# Dense definition ("attention_kernels.py" section 2 ``standard_attention``;
# "lab.py" ``dense``; "flash_attention_numpy.py" ``standard_attention``)
# --------------------------------------------------------------------------
def _dense_rows(q_rows, k, v, sc, causal, q_start):
    """Scores, log-sum-exp and probabilities of a block of whole query rows."""
    s = (q_rows @ k.T) * sc
    if causal:
        s = np.where(causal_mask(q_start, q_rows.shape[0], k.shape[0]), NEG_INF, s)
    m = s.max(axis=1, keepdims=True)
    if not np.all(np.isfinite(m)):
        raise ValueError("a query row sees no key (empty or fully masked row)")
    lse = m[:, 0] + np.log(np.exp(s - m).sum(axis=1))
    p = np.exp(s - lse[:, None])
    return s, lse, p


def attention_dense(q, k, v, scale=None, causal=False, q_start=0):
    """Softmax attention by its definition: S = Q K^T * scale, L = logsumexp_row(S),
    P = exp(S - L), O = P V.  Returns (O, L) with L in natural log.

    Shapes: q (..., Nq, d); k (..., Nk, d); v (..., Nk, dv).  With ``causal``
    the key at position j is visible to query row i iff j <= q_start + i.
    Source: "attention_kernels.py", section 2 ``standard_attention`` (causal
    mask, q_start, log-sum-exp return); the log-sum-exp is taken stably by
    subtracting the row maximum first, as "lab.py" ``dense`` does.
    """
    q, k, v = _as_f64(q, k, v)
    sc = default_scale(q.shape[-1], scale)
    lead = q.shape[:-2]
    nq = q.shape[-2]
    out = np.empty(lead + (nq, v.shape[-1]))
    lse = np.empty(lead + (nq,))
    for h in _heads(q):
        for r0 in range(0, nq, _ROW_CHUNK):
            r1 = min(r0 + _ROW_CHUNK, nq)
            _, l_rows, p = _dense_rows(q[h][r0:r1], k[h], v[h], sc, causal, q_start + r0)
            out[h][r0:r1] = p @ v[h]
            lse[h][r0:r1] = l_rows
    return out, lse


def attention_dense_rows(q, k, v, rows, scale=None, causal=False):
    """Dense-definition output for selected query rows of one head.

    q (Nq, d), k (Nk, d), v (Nk, dv); ``rows`` is a list of query indices
    (q_start = 0).  Same definition as :func:`attention_dense`, evaluated one
    row at a time so that single outputs of a large problem can be checked.
    """
    q, k, v = _as_f64(q, k, v)
    sc = default_scale(q.shape[-1], scale)
    out = np.empty((len(rows), v.shape[-1]))
    lse = np.empty(len(rows))
    for n, i in enumerate(rows):
        kk, vv = (k[: i + 1], v[: i + 1]) if causal else (k, v)
        _, l_row, p = _dense_rows(q[i : i + 1], kk, vv, sc, False, 0)
        out[n] = (p @ vv)[0]
        lse[n] = l_row[0]
    return out, lse


def attention_dense_backward(q, k, v, do, scale=None, causal=False, q_start=0):
    """Gradients of loss = sum(O * dO) through the dense definition.

    With P the softmax probabilities: dV = P^T dO, dP = dO V^T,
    dS = P * (dP - rowsum(P * dP)) (the softmax Jacobian diag(p) - p p^T applied
    to dP, as derived in "attention_kernels.py" section 4), dQ = dS K * scale,
    dK = dS^T Q * scale.  The row sum here is taken over P * dP from its
    definition, not over dO * O, so this path does not depend on a stored O.
    Returns (dQ, dK, dV) in the shapes of (q, k, v).
    """
    q, k, v, do = _as_f64(q, k, v, do)
    sc = default_scale(q.shape[-1], scale)
    nq = q.shape[-2]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for h in _heads(q):
        for r0 in range(0, nq, _ROW_CHUNK):
            r1 = min(r0 + _ROW_CHUNK, nq)
            q_rows, do_rows = q[h][r0:r1], do[h][r0:r1]
            _, _, p = _dense_rows(q_rows, k[h], v[h], sc, causal, q_start + r0)
            dp = do_rows @ v[h].T
            ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))
            dq[h][r0:r1] = (ds @ k[h]) * sc
            dk[h] += (ds.T @ q_rows) * sc
            dv[h] += p.T @ do_rows
    return dq, dk, dv


# --------------------------------------------------------------------------
# Independent row-wise tiled version ("lab.py" ``tiled`` and ``backward``)
# --------------------------------------------------------------------------
def attention_tiled_rowwise(q, k, v, block, scale=None, causal=False):
    """Online-softmax forward, one query row at a time over key tiles of ``block``.

    For each row: m = -inf, l = 0, acc = 0; for each key tile, the tile's scores
    s give m' = max(m, max s), alpha = exp(m - m') (0 while l is still 0),
    e = exp(s - m'), l = alpha*l + sum e, acc = alpha*acc + e V_tile, m = m'.
    Finally O = acc / l and L = m + log l.  Under ``causal`` a tile stops at the
    row's own position and a tile that starts beyond it is skipped whole.
    The last tile may be shorter than ``block``.  Source: "lab.py", ``tiled``.
    Shapes: q (Nq, d), k (Nk, d), v (Nk, dv), a single head.
    """
    if block < 1:
        raise ValueError("block must be >= 1")
    q, k, v = _as_f64(q, k, v)
    sc = default_scale(q.shape[1], scale)
    nk = k.shape[0]
    out = np.zeros((q.shape[0], v.shape[1]))
    lse = np.empty(q.shape[0])
    for i in range(q.shape[0]):
        m, l = NEG_INF, 0.0
        acc = np.zeros(v.shape[1])
        end = i + 1 if causal else nk
        for start in range(0, nk, block):
            stop = min(start + block, nk, end)
            if stop <= start:
                continue
            s = (k[start:stop] @ q[i]) * sc
            m_new = max(m, s.max())
            alpha = np.exp(m - m_new) if l > 0.0 else 0.0
            e = np.exp(s - m_new)
            l = alpha * l + e.sum()
            acc = alpha * acc + e @ v[start:stop]
            m = m_new
        out[i] = acc / l
        lse[i] = m + np.log(l)
    return out, lse


def attention_tiled_rowwise_backward(q, k, v, out, lse, do, block, scale=None, causal=False):
    """Row-wise tiled gradient that recomputes P from the stored log-sum-exp.

    D_i = dO_i . O_i once per row; then per key tile P = exp(s - L_i),
    dP = V_tile dO_i, dS = P * (dP - D_i), dQ_i += dS K_tile * scale,
    dK_tile += dS Q_i * scale, dV_tile += P dO_i.  Source: "lab.py", ``backward``
    (which is the row-wise form of "attention_kernels.py" section 4).
    """
    if block < 1:
        raise ValueError("block must be >= 1")
    q, k, v, out, lse, do = _as_f64(q, k, v, out, lse, do)
    sc = default_scale(q.shape[1], scale)
    nk = k.shape[0]
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    row_dot = (do * out).sum(axis=1)
    for i in range(q.shape[0]):
        end = i + 1 if causal else nk
        for start in range(0, nk, block):
            stop = min(start + block, nk, end)
            if stop <= start:
                continue
            p = np.exp((k[start:stop] @ q[i]) * sc - lse[i])
            dp = v[start:stop] @ do[i]
            ds = p * (dp - row_dot[i])
            dq[i] += (ds @ k[start:stop]) * sc
            dk[start:stop] += np.outer(ds, q[i]) * sc
            dv[start:stop] += np.outer(p, do[i])
    return dq, dk, dv


# --------------------------------------------------------------------------
# Block-wise loop with the page's counters ("attention_kernels.py" §3, §4, §6)
# --------------------------------------------------------------------------
def _bump(stats, key, n):
    if stats is not None:
        stats[key] = stats.get(key, 0) + int(n)


def attention_flash_blocked(q, k, v, br, bc, scale=None, causal=False, stats=None, rescale_margin=0.0):
    """Online softmax over blocks: query blocks of ``br`` rows against key blocks of ``bc`` keys.

    Query blocks outer, key blocks inner.  Under ``causal`` a key block whose first
    key lies after the query block's last row (j0 > i1 - 1) is skipped whole; the
    other blocks mask keys after each row to -inf.  Per computed block, with s the
    block's scores: m_new = max(m, rowmax s), alpha = exp(m - m_new) (0 while m is
    still -inf), p = exp(s - m_new), l = alpha l + rowsum p, acc = alpha acc + p V_j,
    m = m_new.  Finally O_i = acc / l and L_i = m + log l.  Blocks may be uneven
    at the end.

    ``stats`` (a dict) receives the page's counters: "tiles" (blocks computed),
    "skipped" (blocks skipped under causality) and "rescales" (rows of a computed
    block whose running max grew from a finite value).  ``rescale_margin`` is not
    on the page (default 0): a growth counts only when m_new > m + margin, so that
    a test can bracket a count taken in another precision.
    Source: "attention_kernels.py", section 3 ``flash_forward``.  Single head:
    q (Nq, d), k (Nk, d), v (Nk, dv).
    """
    if br < 1 or bc < 1:
        raise ValueError("block sizes must be >= 1")
    q, k, v = _as_f64(q, k, v)
    sc = default_scale(q.shape[1], scale)
    nq, nk = q.shape[0], k.shape[0]
    out = np.empty((nq, v.shape[1]))
    lse = np.empty(nq)
    for i0 in range(0, nq, br):
        i1 = min(i0 + br, nq)
        m = np.full(i1 - i0, NEG_INF)
        l = np.zeros(i1 - i0)
        acc = np.zeros((i1 - i0, v.shape[1]))
        for j0 in range(0, nk, bc):
            j1 = min(j0 + bc, nk)
            if causal and j0 > i1 - 1:
                _bump(stats, "skipped", 1)
                continue
            s = (q[i0:i1] @ k[j0:j1].T) * sc
            if causal:
                s = np.where(causal_mask(i0, i1 - i0, j1 - j0, k_start=j0), NEG_INF, s)
            m_new = np.maximum(m, s.max(axis=1))
            finite = np.isfinite(m)
            alpha = np.where(finite, np.exp(np.where(finite, m, 0.0) - np.where(finite, m_new, 0.0)), 0.0)
            p = np.exp(s - np.where(np.isfinite(m_new), m_new, 0.0)[:, None])
            l = l * alpha + p.sum(axis=1)
            acc = acc * alpha[:, None] + p @ v[j0:j1]
            _bump(stats, "tiles", 1)
            _bump(stats, "rescales", np.count_nonzero(finite & (m_new > np.where(finite, m, 0.0) + rescale_margin)))
            m = m_new
        out[i0:i1] = acc / l[:, None]
        lse[i0:i1] = m + np.log(l)
    return out, lse


def attention_flash_blocked_backward(q, k, v, out, lse, do, br, bc, scale=None, causal=False, stats=None):
    """Recompute backward over blocks: key blocks outer, query blocks inner.

    D = rowsum(dO * O).  For key block j and query block i (skipped whole under
    causality when j0 > i1 - 1): P = exp(S - L_i) with future keys masked,
    dV_j += P^T dO_i, dP = dO_i V_j^T, dS = P * (dP - D_i), dQ_i += dS K_j * scale,
    dK_j += dS^T Q_i * scale.  ``stats`` receives the page's "dq_atomic_adds":
    (i1 - i0) * d per computed block, the dQ elements a GPU adds atomically.
    Source: "attention_kernels.py", section 4 ``flash_backward``.  Single head.
    """
    if br < 1 or bc < 1:
        raise ValueError("block sizes must be >= 1")
    q, k, v, out, lse, do = _as_f64(q, k, v, out, lse, do)
    sc = default_scale(q.shape[1], scale)
    nq, nk = q.shape[0], k.shape[0]
    row_dot = (do * out).sum(axis=1)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for j0 in range(0, nk, bc):
        j1 = min(j0 + bc, nk)
        for i0 in range(0, nq, br):
            i1 = min(i0 + br, nq)
            if causal and j0 > i1 - 1:
                continue
            s = (q[i0:i1] @ k[j0:j1].T) * sc
            if causal:
                s = np.where(causal_mask(i0, i1 - i0, j1 - j0, k_start=j0), NEG_INF, s)
            p = np.exp(s - lse[i0:i1, None])
            dv[j0:j1] += p.T @ do[i0:i1]
            dp = do[i0:i1] @ v[j0:j1].T
            ds = p * (dp - row_dot[i0:i1, None])
            dq[i0:i1] += (ds @ k[j0:j1]) * sc
            dk[j0:j1] += (ds.T @ q[i0:i1]) * sc
            _bump(stats, "dq_atomic_adds", (i1 - i0) * q.shape[1])
    return dq, dk, dv


def attention_fa1_keymajor(q, k, v, br, bc, scale=None, causal=False):
    """The first algorithm's loop order: key blocks outer, query blocks inner.

    The running output O, maximum m and sum r of every query row live outside the
    loops and are repaired at each visit: for key block j and query block i, with
    the block's scores s, m~ = rowmax s, p~ = exp(s - m~), r~ = rowsum p~;
    m' = max(m, m~), r' = e^(m - m') r + e^(m~ - m') r~, and
    O = (e^(m - m') r / r') O + e^(m~ - m') (p~ V_j) / r'; then m, r = m', r'.  O is
    normalised after every visit.  Rows whose scores in a block are all masked take
    nothing from it (their m~ is -inf).  Returns O and L = m + log r.
    Source: "flash_attention_numpy.py" ``flash_attention_tier1`` (unscaled, no
    mask); the scale and the causal skip and mask follow "attention_kernels.py"
    section 3.  Single head: q (N, d), k (N, d), v (N, dv).
    """
    if br < 1 or bc < 1:
        raise ValueError("block sizes must be >= 1")
    q, k, v = _as_f64(q, k, v)
    sc = default_scale(q.shape[1], scale)
    n = q.shape[0]
    out = np.zeros((n, v.shape[1]))
    m = np.full(n, NEG_INF)
    r = np.zeros(n)
    for j0 in range(0, n, bc):
        j1 = min(j0 + bc, n)
        for i0 in range(0, n, br):
            i1 = min(i0 + br, n)
            if causal and j0 > i1 - 1:
                continue
            s = (q[i0:i1] @ k[j0:j1].T) * sc
            if causal:
                s = np.where(causal_mask(i0, i1 - i0, j1 - j0, k_start=j0), NEG_INF, s)
            m_t = s.max(axis=1)
            seen = np.isfinite(m_t)  # rows with a visible key in this block
            p_t = np.where(seen[:, None], np.exp(s - np.where(seen, m_t, 0.0)[:, None]), 0.0)
            r_t = p_t.sum(axis=1)
            m_old, r_old = m[i0:i1], r[i0:i1]
            m_new = np.maximum(m_old, m_t)
            fin_new = np.isfinite(m_new)
            base = np.where(fin_new, m_new, 0.0)
            conv_old = np.where(np.isfinite(m_old), np.exp(np.where(np.isfinite(m_old), m_old, 0.0) - base), 0.0)
            conv_new = np.where(seen, np.exp(np.where(seen, m_t, 0.0) - base), 0.0)
            r_new = conv_old * r_old + conv_new * r_t
            safe = np.where(r_new > 0, r_new, 1.0)
            c = np.where(r_new > 0, conv_old * r_old / safe, 0.0)
            pour = conv_new[:, None] * (p_t @ v[j0:j1]) / safe[:, None]
            out[i0:i1] = c[:, None] * out[i0:i1] + pour
            m[i0:i1], r[i0:i1] = m_new, r_new
    return out, m + np.log(r)


def io_flash(n: int, d: int, br: int, kv_cached: bool = False) -> float:
    """Elements the block-wise forward moves to and from device memory.

    Q read once (N d), O written once (N d), L written (N); every query block reads
    all of K and V (2 N d each time, ceil(N / br) times), or once when they stay
    in cache (``kv_cached``), leaving 4 N d + N.
    Source: "attention_kernels.py", section 6 ``io_flash``.
    """
    kv_reads = 2.0 * n * d * (1 if kv_cached else -(-n // br))
    return 2.0 * n * d + kv_reads + n


# --------------------------------------------------------------------------
# Softmax-state algebra and split-KV decoding ("attention_kernels.py" §1, §5)
# --------------------------------------------------------------------------
@dataclass
class SoftmaxState:
    """Summary of a run of scores s_1..s_n with their value rows v_1..v_n.

    m = max s_i, l = sum exp(s_i - m), o = sum exp(s_i - m) v_i, so the run's
    softmax denominator is exp(m) * l and its output is o / l.  The empty run
    is (m=-inf, l=0, o=0), the identity of :func:`merge_states`.
    Source: "attention_kernels.py", section 1 ``SoftmaxState``.
    """

    m: np.ndarray
    l: np.ndarray
    o: np.ndarray


def empty_state(lead_shape, dv) -> SoftmaxState:
    lead_shape = tuple(lead_shape)
    return SoftmaxState(np.full(lead_shape, NEG_INF), np.zeros(lead_shape), np.zeros(lead_shape + (dv,)))


def _safe_base(m):
    # Both runs empty: m = -inf and exp(-inf - (-inf)) would be NaN; any finite
    # base gives the same (empty) result because l and o are then 0.
    return np.where(np.isinf(m), 0.0, m)


def state_of_scores(s, v) -> SoftmaxState:
    """State of one run of scores s (..., n) with values v (..., n, dv).

    Source: "attention_kernels.py", section 1 ``state_of_scores``.
    """
    s, v = _as_f64(s, v)
    m = s.max(axis=-1)
    p = np.exp(s - _safe_base(m)[..., None])
    return SoftmaxState(m, p.sum(axis=-1), p @ v)


def merge_states(a: SoftmaxState, b: SoftmaxState) -> SoftmaxState:
    """a (+) b: m = max(m_a, m_b); each side is rebased by exp(m_side - m);
    l and o combine linearly.  Associative and commutative, with the empty
    state as identity.  Source: "attention_kernels.py", section 1 ``merge_states``.
    """
    m = np.maximum(a.m, b.m)
    base = _safe_base(m)
    ca, cb = np.exp(a.m - base), np.exp(b.m - base)
    return SoftmaxState(m, a.l * ca + b.l * cb, a.o * ca[..., None] + b.o * cb[..., None])


def split_bounds(nk: int, n_split: int) -> list[int]:
    """Segment boundaries round(nk * s / n_split), s = 0..n_split, with Python's
    round-half-to-even taken on the exact rational value.
    Source: "attention_kernels.py", section 5 ``flash_decode``.
    """
    if n_split < 1:
        raise ValueError("n_split must be >= 1")
    return [round(Fraction(nk * s, n_split)) for s in range(n_split + 1)]


def attention_split_decode(q, k, v, n_split, scale=None):
    """Flash-Decoding: split the keys into n_split segments, take each segment's
    state, fold them left to right with merge_states, and return O = o / l.

    q (..., Nq, d), k (..., Nk, d), v (..., Nk, dv); no causal mask (the decoded
    query sees every key).  Empty segments (n_split > Nk) give the empty state.
    Returns (O, L, parts) with L = m + log l in natural log and ``parts`` the
    per-segment states in split order.
    Source: "attention_kernels.py", section 5 ``flash_decode``.
    """
    q, k, v = _as_f64(q, k, v)
    sc = default_scale(q.shape[-1], scale)
    bounds = split_bounds(k.shape[-2], n_split)
    parts = []
    for s in range(n_split):
        j0, j1 = bounds[s], bounds[s + 1]
        if j1 == j0:
            parts.append(empty_state(q.shape[:-1], v.shape[-1]))
            continue
        scores = (q @ np.swapaxes(k[..., j0:j1, :], -1, -2)) * sc
        parts.append(state_of_scores(scores, v[..., j0:j1, :]))
    total = parts[0]
    for part in parts[1:]:
        total = merge_states(total, part)
    return total.o / total.l[..., None], total.m + np.log(total.l), parts
