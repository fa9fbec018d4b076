"""CPU float64 oracle for Reference Sliding Window Attention (R-SWA).

TEST INFRASTRUCTURE ONLY.  This module is the plain, slow, obviously correct
statement of what the R-SWA hot path computes.  Only the tests, the smoke check
and the benchmark's CPU-baseline leg may import it; the product library never
does, and this module imports nothing from the product (no shared kernels,
helpers, constants or layout code).

Sources (web pages on the method; cited by title and section):

* [DD] "Unlimited-OCR deep dive" (ai-news-5min-kr): the R-SWA pseudo-code
  block "N(t) = P U D_n(t)" with the cache-size line
  "C_R-SWA(T) = L_m + min(n, T) <= L_m + n"; the data-flow steps (1)-(4)
  (prefix fixed and always visible; the cache behaves as a queue that pushes
  out the oldest output KV on each new token); the vanilla-SWA paragraph.
* [GN] "Unlimited OCR - Baidu's one-shot long-document parsing model"
  (GeekNews): section "Reference Sliding Window Attention (R-SWA)" (every
  token sees all reference tokens, output attention limited to the previous
  n = 128 tokens; a two-segment window of size m + n), section "KV cache
  management" (cache L_m + min(n, T) <= L_m + n, versus L_m + T for standard
  MHA), section "Model architecture" (queue of capacity m + n; each new token
  evicts the KV of the (m+1)-th entry).

Readings taken where the pages are silent (each is also listed in the design
notes):

R1  The n-token output window includes the current token: output t sees the
    outputs max(0, t-n+1) .. t.  Only this reading keeps the attended cache at
    m + min(n, T) after T appends and the capacity at m + n.
R2  Prefix rows attend causally among themselves (the decoder is a causal LM
    whose standard MHA is being replaced).
R3  Softmax scale 1/sqrt(d); no bias, ALiBi or soft-cap.
R4  Positions are absolute row indices of the concatenated [prefix | outputs]
    sequence; positional encodings are applied by the caller beforehand.
R5  One KV head per query head (standard MHA, the pages' baseline).  As an
    extension beyond the pages, grouped heads (GQA) are supported: with H
    query heads and H_kv key/value heads (H divisible by H_kv), query head h
    reads KV head h // (H / H_kv).

Notation: m = prefix length (L_m), n = output window, T = number of outputs,
L = m + T rows.  Row i < m is a prefix row; row i >= m is output t = i - m.

Parity status: every function here is pinned by the CPU tests (brute-force
queue simulation, library scaled-dot-product attention, closed forms and
special cases).  Values at realistic shapes beyond those invariants are
"parity unpinned" in the sense that the pages print no numeric attention
output to compare with.
"""

from __future__ import annotations

import collections

import numpy as np

__all__ = [
    "visible",
    "visible_indices",
    "row_visible_count",
    "visible_pair_count",
    "cache_len",
    "ring_slot",
    "ring_outputs",
    "RingQueue",
    "attention_rows",
    "kv_head",
    "prefill_attention",
    "prefill_cache",
    "append_kv",
    "decode_step",
    "decode_step_fused",
]


# ---------------------------------------------------------------------------
# The attention set N(t) = P U D_n(t)   ([DD] pseudo-code block; [GN] R-SWA)
# ---------------------------------------------------------------------------

def visible(i: int, j: int, m: int, n: int) -> bool:
    """True iff row i attends to key j.

    Prefix rows (i < m) are causal (R2).  An output row i >= m sees the whole
    prefix P = {0..m-1} and the outputs in the window D_n = {max(m, i-n+1)..i}
    (R1: the window of n includes the row itself).
    """
    if j < 0 or j > i:
        return False
    if i < m:
        return True
    if j < m:
        return True
    return j >= i - n + 1


def visible_indices(i: int, m: int, n: int) -> np.ndarray:
    """Sorted key indices of N(i) as an int64 array."""
    if i < m:
        return np.arange(0, i + 1, dtype=np.int64)
    lo = max(m, i - n + 1)
    return np.concatenate([np.arange(0, m, dtype=np.int64),
                           np.arange(lo, i + 1, dtype=np.int64)])


def row_visible_count(i: int, m: int, n: int) -> int:
    """|N(i)|: i + 1 for a prefix row, m + min(n, t + 1) for output t = i - m."""
    if i < m:
        return i + 1
    return m + min(n, i - m + 1)


def visible_pair_count(m: int, n: int, L: int) -> int:
    """Number of visible (i, j) pairs over rows 0..L-1 of one head."""
    return sum(row_visible_count(i, m, n) for i in range(L))


# ---------------------------------------------------------------------------
# Cache size and the ring of output KV ([DD] cache-size line; [GN] KV cache
# management and model architecture)
# ---------------------------------------------------------------------------

def cache_len(m: int, n: int, T: int) -> int:
    """Tokens held after T outputs: C(T) = L_m + min(n, T)."""
    return m + min(n, T)


def ring_slot(j: int, n: int) -> int:
    """Ring slot of output j (0-based).  The queue's n output entries are kept
    in n slots; the entry evicted by output j is output j - n, which lived in
    the same slot, so the slot of output j is j mod n."""
    return j % n


def ring_outputs(t: int, n: int) -> dict:
    """Slot -> output index held after t appends (outputs max(0,t-n)..t-1)."""
    return {ring_slot(j, n): j for j in range(max(0, t - n), t)}


class RingQueue:
    """The pages' literal queue of capacity m + n.

    Entries are token positions.  The m prefix entries are pushed once and
    never leave; each output push beyond capacity evicts the (m+1)-th entry,
    i.e. the oldest output.  The output part is a deque(maxlen=n).
    """

    def __init__(self, m: int, n: int):
        self.m = m
        self.n = n
        self.prefix = list(range(m))
        self.outputs = collections.deque(maxlen=n)
        self.t = 0

    def push_output(self) -> None:
        self.outputs.append(self.m + self.t)
        self.t += 1

    def contents(self) -> list:
        return self.prefix + list(self.outputs)

    def __len__(self) -> int:
        return len(self.prefix) + len(self.outputs)


# ---------------------------------------------------------------------------
# Masked softmax attention (definition; R3)
# ---------------------------------------------------------------------------

def _attend(q: np.ndarray, K: np.ndarray, V: np.ndarray):
    """softmax(q . K^T / sqrt(d)) @ V in float64, plus the natural-log
    log-sum-exp of the scaled logits."""
    d = q.shape[-1]
    x = (K @ q) / np.sqrt(d)
    mx = x.max()
    w = np.exp(x - mx)
    s = w.sum()
    return (w @ V) / s, mx + np.log(s)


def attention_rows(Q, K, V, m: int, n: int, rows=None):
    """R-SWA attention for one head.

    Q, K, V: [L][d] arrays (any float dtype; converted exactly to float64).
    Returns (O [len(rows)][d], lse [len(rows)]) in float64 for the requested
    rows (all rows by default).
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    L, d = Q.shape
    if rows is None:
        rows = range(L)
    rows = list(rows)
    O = np.empty((len(rows), V.shape[1]), dtype=np.float64)
    lse = np.empty(len(rows), dtype=np.float64)
    for r, i in enumerate(rows):
        idx = visible_indices(i, m, n)
        O[r], lse[r] = _attend(Q[i], K[idx], V[idx])
    return O, lse


def kv_head(h: int, H: int, Hkv: int) -> int:
    """KV head read by query head h (R5)."""
    return h // (H // Hkv)


def prefill_attention(Q, K, V, m: int, n: int, rows=None):
    """R-SWA prefill for token-major inputs Q [L][H][d], K, V [L][H_kv][d].

    Returns (O [R][H][d], lse [R][H]) for the requested rows R (default all).
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K)
    V = np.asarray(V)
    L, H, d = Q.shape
    Hkv = K.shape[1]
    rows = list(range(L)) if rows is None else list(rows)
    O = np.empty((len(rows), H, V.shape[2]), dtype=np.float64)
    lse = np.empty((len(rows), H), dtype=np.float64)
    for h in range(H):
        g = kv_head(h, H, Hkv)
        O[:, h], lse[:, h] = attention_rows(Q[:, h], K[:, g], V[:, g], m, n,
                                            rows)
    return O, lse


# ---------------------------------------------------------------------------
# Cache state transitions ([DD] data-flow steps (2) and (4); [GN] model
# architecture: queue of capacity m + n, evict the (m+1)-th entry)
# ---------------------------------------------------------------------------

def prefill_cache(K, V, m: int, n: int, T: int):
    """State after prefilling m prefix rows and T outputs of one sequence.

    K, V: [m + T][H_kv][d].  Returns dict(Kp, Vp [m][H_kv][d], Kr, Vr
    [n][H_kv][d] with
    never-written slots set to NaN, t = T).
    """
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    H, d = K.shape[1], K.shape[2]
    Kr = np.full((n, H, d), np.nan)
    Vr = np.full((n, H, d), np.nan)
    for slot, j in ring_outputs(T, n).items():
        Kr[slot] = K[m + j]
        Vr[slot] = V[m + j]
    return {"Kp": K[:m].copy(), "Vp": V[:m].copy(), "Kr": Kr, "Vr": Vr, "t": T}


def append_kv(state: dict, k, v, n: int) -> dict:
    """Write output t's k, v ([H_kv][d]) into slot t mod n, then t += 1."""
    t = state["t"]
    Kr = state["Kr"].copy()
    Vr = state["Vr"].copy()
    Kr[ring_slot(t, n)] = np.asarray(k, dtype=np.float64)
    Vr[ring_slot(t, n)] = np.asarray(v, dtype=np.float64)
    return {"Kp": state["Kp"], "Vp": state["Vp"], "Kr": Kr, "Vr": Vr, "t": t + 1}


def decode_step(state: dict, q, n: int):
    """Attend q ([H][d]) over the cache: the prefix plus the filled ring slots
    (query head h reads KV head h // (H / H_kv)).

    The caller appends output t's k, v before decoding q_t, so the row attends
    to itself (R1).  Returns (o [H][d], lse [H]) in float64.
    """
    q = np.asarray(q, dtype=np.float64)
    filled = sorted(ring_outputs(state["t"], n).keys())
    H = q.shape[0]
    Hkv = state["Kr"].shape[1]
    o = np.empty((H, state["Vr"].shape[2]), dtype=np.float64)
    lse = np.empty(H, dtype=np.float64)
    for h in range(H):
        g = kv_head(h, H, Hkv)
        Kc = np.concatenate([state["Kp"][:, g], state["Kr"][filled, g]])
        Vc = np.concatenate([state["Vp"][:, g], state["Vr"][filled, g]])
        o[h], lse[h] = _attend(q[h], Kc, Vc)
    return o, lse


def decode_step_fused(state: dict, q, k, v, n: int):
    """append_kv followed by decode_step; returns (new_state, o, lse)."""
    new_state = append_kv(state, k, v, n)
    o, lse = decode_step(new_state, q, n)
    return new_state, o, lse
