"""Pins of the CPU oracle against facts it does not compute itself.

Each check below is written as a function of the oracle module so that the
mutation test at the end can re-run it against deliberately broken copies of
the oracle and show that a plausible mistake fails at least one pin.

What pins what:
* the mask: a literal simulation of the pages' queue of capacity m + n that
  evicts the (m+1)-th entry on every new output ("Unlimited OCR", GeekNews,
  section "Model architecture"; "Unlimited-OCR deep dive", data-flow step 4),
  exhaustively over small (m, n, T), plus a hand-worked fixture;
* the cache size: the closed form C(T) = L_m + min(n, T) printed on both pages
  and a hand-worked fixture;
* the ring: a physical ring with a wrapping write pointer and a
  ``collections.deque(maxlen=n)``;
* the attention arithmetic: torch's float64 scaled_dot_product_attention (a
  library routine) with the causal flag (R-SWA with n >= T is full causal
  attention) and with a boolean mask taken from the queue simulation;
* special cases with closed forms: constant V gives V, q = 0 with V = I
  reveals the visible set through the output values and gives
  lse = ln |N(i)|;
* decode against prefill: decode step t through the ring equals prefill row
  m + t.
"""

import importlib.util
import math
import os
import sys
import types

import numpy as np
import pytest
import torch

import oracle as ORC

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = os.path.join(HERE, "golden")


# ---------------------------------------------------------------------------
# Independent models
# ---------------------------------------------------------------------------

def queue_simulation(m, n, L):
    """Visible sets by pushing positions into the pages' queue.

    Every position is pushed in order; once outputs start (position >= m) a
    push that takes the queue over capacity m + n removes the (m+1)-th entry.
    The row attends to what the queue holds right after its own push.
    """
    cache, sets = [], []
    for i in range(L):
        cache.append(i)
        if i >= m and len(cache) > m + n:
            del cache[m]
        sets.append(list(cache))
    return sets


def physical_ring(n, t):
    """Slot -> output after t appends, with a write pointer that wraps."""
    slots, ptr = [None] * n, 0
    for j in range(t):
        slots[ptr] = j
        ptr += 1
        if ptr == n:
            ptr = 0
    return {s: j for s, j in enumerate(slots) if j is not None}


def read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def parse_set(s):
    return [int(x) for x in s.split(",")]


# ---------------------------------------------------------------------------
# Pin checks (each takes the oracle module)
# ---------------------------------------------------------------------------

def check_mask_vs_queue(orc):
    for m in range(0, 7):
        for n in range(1, 7):
            for T in range(0, 13):
                L = m + T
                sets = queue_simulation(m, n, L)
                for i in range(L):
                    exp = sets[i]
                    got = orc.visible_indices(i, m, n).tolist()
                    assert got == sorted(exp), (m, n, T, i, got, exp)
                    assert orc.row_visible_count(i, m, n) == len(exp)
                    for j in range(L):
                        assert orc.visible(i, j, m, n) == (j in exp), (m, n, i, j)
                if L:
                    brute = sum(len(s) for s in sets)
                    assert orc.visible_pair_count(m, n, L) == brute


def check_cache_size(orc):
    for m in range(0, 6):
        for n in range(1, 6):
            q = orc.RingQueue(m, n)
            sets = queue_simulation(m, n, m + 20)
            assert orc.cache_len(m, n, 0) == m == len(q)
            for t in range(20):
                q.push_output()
                assert len(q) == orc.cache_len(m, n, t + 1) == len(sets[m + t])
                assert q.contents() == sets[m + t]
    for Lm, n, T, rswa, mha in read_table("cache_size_curve.txt"):
        Lm, n, T = int(Lm), int(n), int(T)
        assert orc.cache_len(Lm, n, T) == int(rswa)
        # n >= T turns R-SWA into the standard cache L_m + T
        assert orc.cache_len(Lm, T + 1, T) == int(mha)


def check_ring(orc):
    for n in range(1, 9):
        dq = __import__("collections").deque(maxlen=n)
        for t in range(0, 3 * n + 5):
            exp = physical_ring(n, t)
            assert orc.ring_outputs(t, n) == exp, (n, t)
            assert sorted(exp.values()) == list(dq)
            for j in exp.values():
                assert exp[orc.ring_slot(j, n)] == j
            dq.append(t)


def check_mask_golden(orc):
    m, n = 3, 2
    for row, kind, rswa, swa, causal in read_table("rswa_mask_m3_n2_T5.txt"):
        i = int(row)
        assert orc.visible_indices(i, m, n).tolist() == parse_set(rswa)
        # vanilla SWA = R-SWA with an empty prefix
        assert orc.visible_indices(i, 0, n).tolist() == parse_set(swa)
        # full causal = R-SWA with a window no smaller than the outputs
        assert orc.visible_indices(i, m, 100).tolist() == parse_set(causal)


def _sdpa(Q, K, V, mask=None, causal=False):
    """torch float64 SDPA on [L][H][d] arrays; returns [L][H][d]."""
    q = torch.from_numpy(Q).permute(1, 0, 2)[None]
    k = torch.from_numpy(K).permute(1, 0, 2)[None]
    v = torch.from_numpy(V).permute(1, 0, 2)[None]
    am = None if mask is None else torch.from_numpy(mask)
    o = torch.nn.functional.scaled_dot_product_attention(
        q, k, v, attn_mask=am, is_causal=causal)
    return o[0].permute(1, 0, 2).numpy()


def check_causal_sdpa(orc):
    rng = np.random.default_rng(1)
    for (m, T, H, d, dv) in [(5, 32, 3, 16, 16), (0, 21, 2, 8, 8),
                             (17, 0, 1, 24, 24), (3, 12, 2, 16, 5)]:
        L = m + T
        Q = rng.standard_normal((L, H, d))
        K = rng.standard_normal((L, H, d))
        V = rng.standard_normal((L, H, dv))
        ref = _sdpa(Q, K, V, causal=True)
        got, _ = orc.prefill_attention(Q, K, V, m, max(T, 1))
        np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def check_masked_sdpa(orc):
    rng = np.random.default_rng(2)
    for (m, n, T, H, d) in [(0, 4, 30, 2, 16), (7, 3, 25, 2, 16),
                            (4, 1, 9, 1, 8), (11, 5, 40, 3, 32)]:
        L = m + T
        sets = queue_simulation(m, n, L)
        mask = np.zeros((L, L), dtype=bool)
        for i, s in enumerate(sets):
            mask[i, s] = True
        Q = 2.0 * rng.standard_normal((L, H, d))
        K = rng.standard_normal((L, H, d))
        V = rng.standard_normal((L, H, d))
        ref = _sdpa(Q, K, V, mask=mask)
        got, lse = orc.prefill_attention(Q, K, V, m, n)
        np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)
        # lse against torch.logsumexp of the masked logits
        x = torch.einsum("ihd,jhd->hij", torch.from_numpy(Q),
                         torch.from_numpy(K)) / math.sqrt(d)
        x = x.masked_fill(~torch.from_numpy(mask)[None], float("-inf"))
        ref_lse = torch.logsumexp(x, dim=-1).permute(1, 0).numpy()
        np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


def check_identity_values(orc):
    for (m, n, T) in [(4, 3, 9), (0, 2, 7), (6, 1, 6), (2, 8, 5)]:
        L = m + T
        d = L + 3
        sets = queue_simulation(m, n, L)
        Q = np.zeros((L, 1, d))
        K = np.random.default_rng(3).standard_normal((L, 1, d))
        V = np.zeros((L, 1, d))
        V[:, 0, :L] = np.eye(L)
        O, lse = orc.prefill_attention(Q, K, V, m, n)
        for i, s in enumerate(sets):
            exp = np.zeros(d)
            exp[s] = 1.0 / len(s)
            np.testing.assert_allclose(O[i, 0], exp, rtol=0, atol=1e-15)
            assert abs(lse[i, 0] - math.log(len(s))) < 1e-13


def check_constant_v(orc):
    rng = np.random.default_rng(4)
    m, n, T, H, d = 5, 3, 11, 2, 8
    L = m + T
    c = rng.standard_normal((H, d))
    V = np.broadcast_to(c, (L, H, d)).copy()
    O, _ = orc.prefill_attention(3 * rng.standard_normal((L, H, d)),
                                 rng.standard_normal((L, H, d)), V, m, n)
    np.testing.assert_allclose(O, np.broadcast_to(c, O.shape), rtol=0,
                               atol=1e-13)


def check_decode_equals_prefill_row(orc):
    rng = np.random.default_rng(5)
    for (m, n, T, H, d) in [(6, 4, 13, 2, 8), (0, 3, 9, 1, 4),
                            (9, 16, 10, 2, 8), (3, 1, 5, 1, 4)]:
        L = m + T
        Q = rng.standard_normal((L, H, d))
        K = rng.standard_normal((L, H, d))
        V = rng.standard_normal((L, H, d))
        O, lse = orc.prefill_attention(Q, K, V, m, n)
        state = orc.prefill_cache(K[:m], V[:m], m, n, 0)
        for t in range(T):
            state, o, l = orc.decode_step_fused(state, Q[m + t], K[m + t],
                                                V[m + t], n)
            np.testing.assert_allclose(o, O[m + t], rtol=0, atol=1e-12)
            np.testing.assert_allclose(l, lse[m + t], rtol=0, atol=1e-12)
            assert state["t"] == t + 1
        # prefilling all T outputs gives the same ring as T appends
        direct = orc.prefill_cache(K, V, m, n, T)
        filled = sorted(orc.ring_outputs(T, n))
        np.testing.assert_array_equal(direct["Kr"][filled], state["Kr"][filled])
        np.testing.assert_array_equal(direct["Vr"][filled], state["Vr"][filled])


def check_gqa_repeated_kv(orc):
    """Grouped heads equal standard MHA with each KV head repeated for its
    group of query heads (torch SDPA on explicitly repeated K, V)."""
    rng = np.random.default_rng(6)
    for (m, n, T, H, Hkv, d) in [(6, 4, 20, 4, 2, 8), (3, 2, 11, 6, 3, 16),
                                 (5, 3, 9, 4, 1, 8)]:
        L = m + T
        sets = queue_simulation(m, n, L)
        mask = np.zeros((L, L), dtype=bool)
        for i, st in enumerate(sets):
            mask[i, st] = True
        Q = rng.standard_normal((L, H, d))
        K = rng.standard_normal((L, Hkv, d))
        V = rng.standard_normal((L, Hkv, d))
        Kr = np.repeat(K, H // Hkv, axis=1)
        Vr = np.repeat(V, H // Hkv, axis=1)
        ref = _sdpa(Q, Kr, Vr, mask=mask)
        got, _ = orc.prefill_attention(Q, K, V, m, n)
        np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)
        # and through the cache: decode step t equals prefill row m + t
        state = orc.prefill_cache(K[:m], V[:m], m, n, 0)
        for t in range(T):
            state, o, _ = orc.decode_step_fused(state, Q[m + t], K[m + t],
                                                V[m + t], n)
            np.testing.assert_allclose(o, got[m + t], rtol=0, atol=1e-12)


PINS = [check_mask_vs_queue, check_cache_size, check_ring, check_mask_golden,
        check_causal_sdpa, check_masked_sdpa, check_identity_values,
        check_constant_v, check_decode_equals_prefill_row, check_gqa_repeated_kv]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(ORC)


def test_pair_count_closed_form():
    # multipage workload: 286,712,400 visible pairs per head
    m, n, T = 10272, 128, 22496
    assert ORC.visible_pair_count(m, n, m + T) == 286_712_400
    closed = m * (m + 1) // 2 + T * m + sum(min(n, t + 1) for t in range(T))
    assert closed == 286_712_400


# ---------------------------------------------------------------------------
# Mutation test: broken copies of the oracle must fail some pin
# ---------------------------------------------------------------------------

MUTATIONS = [
    ("window drops self", "return j >= i - n + 1", "return j >= i - n + 2"),
    ("window one too wide", "return j >= i - n + 1", "return j >= i - n"),
    ("indices window off", "lo = max(m, i - n + 1)", "lo = max(m, i - n)"),
    ("prefix not exempt", "    if j < m:\n        return True\n", ""),
    ("bidirectional prefix", "if j < 0 or j > i:", "if j < 0 or (j > i and i >= m):"),
    ("scale 1/d", "x = (K @ q) / np.sqrt(d)", "x = (K @ q) / d"),
    ("no scale", "x = (K @ q) / np.sqrt(d)", "x = (K @ q)"),
    ("lse without max", "return (w @ V) / s, mx + np.log(s)",
     "return (w @ V) / s, np.log(s)"),
    ("ring slot shifted", "return j % n", "return (j + 1) % n"),
    ("cache len uses T", "return m + min(n, T)", "return m + T"),
    ("row count off", "return m + min(n, i - m + 1)", "return m + min(n, i - m)"),
    ("append before slot read", "Kr[ring_slot(t, n)] = np.asarray(k, dtype=np.float64)",
     "Kr[ring_slot(t + 1, n)] = np.asarray(k, dtype=np.float64)"),
    ("decode skips newest", "filled = sorted(ring_outputs(state[\"t\"], n).keys())",
     "filled = sorted(ring_outputs(state[\"t\"] - 1, n).keys())"),
    ("values transposed", "return (w @ V) / s, mx + np.log(s)",
     "return (w @ V[:, ::-1]) / s, mx + np.log(s)"),
    ("kv head modulo", "return h // (H // Hkv)", "return h % Hkv"),
]


def _mutant(src, old, new):
    assert old in src, old
    mod = types.ModuleType("oracle_mutant")
    exec(compile(src.replace(old, new, 1), "oracle_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_mutation_is_caught(name, old, new):
    path = os.path.join(os.path.dirname(HERE), "oracle", "rswa_oracle.py")
    with open(path) as f:
        src = f.read()
    mod = _mutant(src, old, new)
    failed = []
    for pin in PINS:
        try:
            pin(mod)
        except Exception:  # AssertionError or a shape error
            failed.append(pin.__name__)
    assert failed, f"mutation '{name}' passed every pin"
