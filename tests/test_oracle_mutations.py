"""The pins catch plausible mistakes: each case plants one mistake in a copy of the
oracle's source (CPU only, in memory) and checks that a pin check then fails."""
import math
import types
from pathlib import Path

import numpy as np
import pytest
import scipy.special

from tests.golden.fixtures import load
from tests.test_oracle_blocked import _block_any, _brute_rescales, _visible

SRC = (Path(__file__).resolve().parent.parent / "oracle" / "attention.py").read_text()


def _mutant(old: str, new: str):
    assert SRC.count(old) >= 1, old
    mod = types.ModuleType("oracle_mutant")
    exec(compile(SRC.replace(old, new, 1), "oracle_mutant", "exec"), mod.__dict__)
    return mod


def _pins_pass(o) -> bool:
    """A compact run of the forward, backward and decode pins against module ``o``."""
    try:
        rng = np.random.default_rng(3)
        g = load("anchor_n3_d2.txt")
        e = math.e
        out, lse = o.attention_dense(g["Q"], g["K"], g["V"], scale=1.0)
        np.testing.assert_allclose(out[0], [(e + e * e) / (1 + e + e * e), (1 + e * e) / (1 + e + e * e)], atol=1e-12)
        np.testing.assert_allclose(lse[0], math.log(1 + e + e * e), atol=1e-12)
        out, lse = o.attention_dense(g["Q"], g["K"], g["V"], scale=1.0, causal=True)
        np.testing.assert_allclose(out[:2], [[1, 0], [0.5, 0.5]], atol=1e-12)
        q, k, v, do = (rng.normal(size=(6, 4)) for _ in range(4))
        s = np.einsum("id,jd->ij", q, k) / 2.0
        ref_o = scipy.special.softmax(s, axis=1) @ v
        out, lse = o.attention_dense(q, k, v)
        np.testing.assert_allclose(out, ref_o, atol=1e-12)
        for causal in (False, True):
            d_o, d_l = o.attention_dense(q, k, v, causal=causal)
            for block in (1, 2, 4):
                t_o, t_l = o.attention_tiled_rowwise(q, k, v, block, causal=causal)
                np.testing.assert_allclose(t_o, d_o, atol=1e-12)
                np.testing.assert_allclose(t_l, d_l, atol=1e-12)
            h = 1e-5
            fd = []
            for arr in (q, k, v):
                gr = np.zeros_like(arr)
                for idx in np.ndindex(arr.shape):
                    old = arr[idx]
                    arr[idx] = old + h
                    plus = np.sum(o.attention_dense(q, k, v, causal=causal)[0] * do)
                    arr[idx] = old - h
                    minus = np.sum(o.attention_dense(q, k, v, causal=causal)[0] * do)
                    arr[idx] = old
                    gr[idx] = (plus - minus) / (2 * h)
                fd.append(gr)
            for a, b in zip(o.attention_dense_backward(q, k, v, do, causal=causal), fd):
                np.testing.assert_allclose(a, b, atol=2e-8, rtol=2e-6)
            t_o, t_l = o.attention_tiled_rowwise(q, k, v, 2, causal=causal)
            for a, b in zip(o.attention_tiled_rowwise_backward(q, k, v, t_o, t_l, do, 2, causal=causal), fd):
                np.testing.assert_allclose(a, b, atol=2e-8, rtol=2e-6)
        # the block-wise loop with its counters ("attention_kernels.py" sections 3, 4, 6)
        qb, kb, vb, dob = (rng.normal(size=(11, 4)) for _ in range(4))
        for causal in (False, True):
            d_o, d_l = o.attention_dense(qb, kb, vb, causal=causal)
            d_g = o.attention_dense_backward(qb, kb, vb, dob, causal=causal)
            for br, bc in ((2, 3), (4, 2), (3, 3)):
                st, sb = {}, {}
                b_o, b_l = o.attention_flash_blocked(qb, kb, vb, br, bc, causal=causal, stats=st)
                np.testing.assert_allclose(b_o, d_o, atol=1e-12)
                np.testing.assert_allclose(b_l, d_l, atol=1e-12)
                b_g = o.attention_flash_blocked_backward(qb, kb, vb, d_o, d_l, dob, br, bc, causal=causal, stats=sb)
                for a, b in zip(b_g, d_g):
                    np.testing.assert_allclose(a, b, atol=1e-11)
                computed = _block_any(_visible(11, causal), br, bc)
                assert st.get("tiles", 0) == int(computed.sum())
                assert st.get("skipped", 0) == int(computed.size - computed.sum())
                assert st.get("rescales", 0) == _brute_rescales(qb, kb, br, bc, causal)
                rows = np.array([min(br, 11 - a * br) for a in range(computed.shape[0])])
                assert sb["dq_atomic_adds"] == int((computed.sum(axis=1) * rows).sum()) * 4
        assert o.io_flash(8, 2, 4) == 104 and o.io_flash(8, 2, 4, kv_cached=True) == 72
        # the key-major loop order (first algorithm)
        for causal in (False, True):
            d_o, d_l = o.attention_dense(qb, kb, vb, causal=causal)
            for br, bc in ((2, 3), (4, 4)):
                k_o, k_l = o.attention_fa1_keymajor(qb, kb, vb, br, bc, causal=causal)
                np.testing.assert_allclose(k_o, d_o, atol=1e-12)
                np.testing.assert_allclose(k_l, d_l, atol=1e-12)
        # a query block at the end of a square causal problem (general q_start)
        qs_o, qs_l = o.attention_dense(qb[7:], kb, vb, causal=True, q_start=7)
        sq_o, sq_l = o.attention_dense(qb, kb, vb, causal=True)
        np.testing.assert_allclose(qs_o, sq_o[7:], atol=1e-13)
        np.testing.assert_allclose(qs_l, sq_l[7:], atol=1e-13)
        dob4 = np.zeros_like(dob)
        dob4[7:] = dob[7:]
        g_block = o.attention_dense_backward(qb[7:], kb, vb, dob[7:], causal=True, q_start=7)
        g_square = o.attention_dense_backward(qb, kb, vb, dob4, causal=True)
        np.testing.assert_allclose(g_block[0], g_square[0][7:], atol=1e-12)  # dQ of the block's rows
        np.testing.assert_allclose(g_block[1], g_square[1], atol=1e-12)      # dK
        np.testing.assert_allclose(g_block[2], g_square[2], atol=1e-12)      # dV
        assert o.split_bounds(10, 4) == [0, 2, 5, 8, 10]
        qd, kd, vd = rng.normal(size=(1, 8)), rng.normal(size=(13, 8)), rng.normal(size=(13, 8))
        ref_o, ref_l = o.attention_dense(qd, kd, vd)
        for n_split in (1, 3, 20):
            dec_o, dec_l, parts = o.attention_split_decode(qd, kd, vd, n_split)
            np.testing.assert_allclose(dec_o, ref_o, atol=1e-12)
            np.testing.assert_allclose(dec_l, ref_l, atol=1e-12)
            bounds = o.split_bounds(13, n_split)
            for si, part in enumerate(parts):  # an empty segment is the identity (-inf, 0, 0)
                if bounds[si + 1] == bounds[si]:
                    assert np.all(np.isneginf(part.m)) and np.all(part.l == 0) and np.all(part.o == 0)
        # a state's m is its run's max; merging two empty states gives the empty state
        sc = rng.normal(scale=3.0, size=(3, 10))
        st = o.state_of_scores(sc, rng.normal(size=(10, 4)))
        np.testing.assert_array_equal(st.m, sc.max(axis=1))
        e = o.empty_state((3,), 4)
        ee = o.merge_states(e, e)
        assert np.all(np.isneginf(ee.m)) and np.all(ee.l == 0) and np.all(ee.o == 0)
    except (AssertionError, ValueError, FloatingPointError):
        return False
    return True


def test_unmodified_oracle_passes():
    assert _pins_pass(_mutant("NEG_INF = -np.inf", "NEG_INF = -np.inf"))


MUTATIONS = [
    ("dropped scale", "s = (q_rows @ k.T) * sc", "s = (q_rows @ k.T)"),
    ("causal off by one", "return kpos > qpos", "return kpos > qpos + 1"),
    ("lse without max", "lse = m[:, 0] + np.log(", "lse = 0 * m[:, 0] + np.log("),
    ("no accumulator rescale", "acc = alpha * acc + e @ v[start:stop]", "acc = acc + e @ v[start:stop]"),
    ("no denominator rescale", "l = alpha * l + e.sum()", "l = l + e.sum()"),
    ("transposed value rows", "out[h][r0:r1] = p @ v[h]", "out[h][r0:r1] = p @ v[h][::-1]"),
    ("dropped D term", "ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))", "ds = p * dp"),
    ("dK from dS not dS^T", "dk[h] += (ds.T @ q_rows) * sc", "dk[h] += (ds @ q_rows) * sc"),
    ("wrong sign of D (tiled)", "ds = p * (dp - row_dot[i])", "ds = p * (dp + row_dot[i])"),
    ("dV scaled", "dv[start:stop] += np.outer(p, do[i])", "dv[start:stop] += np.outer(p, do[i]) * sc"),
    ("merge uses wrong rebase", "a.l * ca + b.l * cb", "a.l * ca + b.l * ca"),
    ("floor split bounds", "round(Fraction(nk * s, n_split))", "int(Fraction(nk * s, n_split))"),
    ("decode drops last segment", "for part in parts[1:]:", "for part in parts[1:-1]:"),
    ("blocked: no accumulator rescale", "acc = acc * alpha[:, None] + p @ v[j0:j1]", "acc = acc + p @ v[j0:j1]"),
    ("blocked: causal skip one block late", "if causal and j0 > i1 - 1:\n                _bump", "if causal and j0 > i1:\n                _bump"),
    ("blocked: rescales counted from -inf", "np.count_nonzero(finite & (m_new >", "np.count_nonzero((m_new >"),
    ("blocked backward: D term dropped", "ds = p * (dp - row_dot[i0:i1, None])", "ds = p * dp"),
    ("blocked backward: dq adds miss rows", "(i1 - i0) * q.shape[1])", "q.shape[1])"),
    ("io_flash: K and V always cached", "(1 if kv_cached else -(-n // br))", "1"),
    ("key-major: old sum not repaired", "r_new = conv_old * r_old + conv_new * r_t", "r_new = r_old + conv_new * r_t"),
    ("key-major: blend not diluted", "c = np.where(r_new > 0, conv_old * r_old / safe, 0.0)", "c = np.where(r_new > 0, conv_old, 0.0)"),
    ("key-major: newcomer not converted", "pour = conv_new[:, None] * (p_t @ v[j0:j1]) / safe[:, None]", "pour = (p_t @ v[j0:j1]) / safe[:, None]"),
    ("dense backward: dQ without scale", "dq[h][r0:r1] = (ds @ k[h]) * sc", "dq[h][r0:r1] = ds @ k[h]"),
    ("dense backward: dV from P not P^T", "dv[h] += p.T @ do_rows", "dv[h] += p[:, :do_rows.shape[0]].T @ do_rows[:p.shape[0]]"),
    ("tiled: rescale sign flipped", "alpha = np.exp(m - m_new) if l > 0.0 else 0.0", "alpha = np.exp(m_new - m) if l > 0.0 else 0.0"),
    ("tiled: LSE in base 2", "lse[i] = m + np.log(l)", "lse[i] = m + np.log2(l)"),
    ("tiled: exponent not shifted by the max", "e = np.exp(s - m_new)", "e = np.exp(s) * 0 + np.exp(s - m)"),
    ("tiled backward: dQ without scale", "dq[i] += (ds @ k[start:stop]) * sc", "dq[i] += ds @ k[start:stop]"),
    ("state: m from the first score", "m = s.max(axis=-1)", "m = s[..., 0]"),
    ("decode: empty segment given a zero max", "parts.append(empty_state(q.shape[:-1], v.shape[-1]))",
     "parts.append(SoftmaxState(np.zeros(q.shape[:-1]), np.zeros(q.shape[:-1]), np.zeros(q.shape[:-1] + (v.shape[-1],))))"),
    ("merge: guarded base dropped", "return np.where(np.isinf(m), 0.0, m)", "return m"),
    ("mask ignores q_start", "qpos = np.arange(q_start, q_start + nq)[:, None]", "qpos = np.arange(0, nq)[:, None]"),
    ("dense backward ignores q_start", "_, _, p = _dense_rows(q_rows, k[h], v[h], sc, causal, q_start + r0)",
     "_, _, p = _dense_rows(q_rows, k[h], v[h], sc, causal, r0)"),
]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(name, old, new):
    with np.errstate(all="ignore"):
        assert not _pins_pass(_mutant(old, new)), name
