"""GPU parity: the CUDA path through the C ABI against the CPU float64 oracle.

Tolerances (fixed for this method): float32 caches max |err| <= 1e-4; bf16
inputs with float32 accumulation max |err| <= 2e-2 and mean |err| <= 5e-3.
Ring indices, t_b and cache sizes must match bit-exactly.  Inputs come from
the seeded generators in ``workloads``; the oracle receives exact float64
copies of the same values.
"""

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

F32_TOL = 1e-4
BF16_MAX, BF16_MEAN = 2e-2, 5e-3


def tdt(dtype):
    return torch.float32 if dtype == 0 else torch.bfloat16


def f64(t):
    return t.detach().double().cpu().numpy()


def _worst(got, ref, err):
    """Where the largest error sits, with both values there."""
    idx = np.unravel_index(int(np.nanargmax(np.where(np.isfinite(err), err, np.inf))),
                           err.shape)
    return f"at {tuple(int(i) for i in idx)}: got {float(got[idx]):.6g}, oracle {float(ref[idx]):.6g}"


def assert_close(got, ref, dtype, what=""):
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - ref)
    assert np.isfinite(err).all(), f"{what}: non-finite output {_worst(got, ref, err)}"
    if dtype == 0:
        assert err.max() <= F32_TOL, f"{what}: max {err.max():.3e} {_worst(got, ref, err)}"
    else:
        assert err.max() <= BF16_MAX, f"{what}: max {err.max():.3e} {_worst(got, ref, err)}"
        assert err.mean() <= BF16_MEAN, f"{what}: mean {err.mean():.3e}"


def make_seq(m_list, T, H, d, dtype, seed, std=1.0):
    """Packed token-major Q, K, V for sequences with prefixes m_list."""
    rows = sum(m + T for m in m_list)
    return workloads.qkv(rows, H, d, seed, std, tdt(dtype))


def oracle_prefill(Q, K, V, m_list, T, n, rows=None):
    """Oracle rows per sequence; returns list of (O, lse) arrays."""
    out, off = [], 0
    for m in m_list:
        L = m + T
        sl = slice(off, off + L)
        out.append(oracle.prefill_attention(f64(Q[sl]), f64(K[sl]), f64(V[sl]),
                                            m, n, rows))
        off += L
    return out


# ---------------------------------------------------------------------------
# tiny float32 workload: prefill of the prefix, then 64 append+decode steps
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("fused", [False, True])
def test_tiny_f32_decode_loop(cuda_lib, fused):
    rswa = cuda_lib
    w = workloads.WORKLOADS["tiny_f32"]
    B, H, d, m, n, T = w.batch, w.heads, w.head_dim, w.m, w.n, w.T
    Q, K, V = make_seq([m], T, H, d, 0, seed=0)
    ref, ref_lse = oracle.prefill_attention(f64(Q), f64(K), f64(V), m, n)
    cache = rswa.RswaCache(m, n, H, d, B, rswa.RSWA_F32)
    Qd, Kd, Vd = Q.cuda(), K.cuda(), V.cuda()
    cache.prefill(None, Kd[:m].contiguous(), Vd[:m].contiguous(), None, [m], 0)
    assert cache.cache_len(0) == oracle.cache_len(m, n, 0)
    Ks, Vs = cache.slabs()
    state = oracle.prefill_cache(f64(K[:m]), f64(V[:m]), m, n, 0)
    for t in range(T):
        q, k, v = (x[m + t][None].contiguous() for x in (Qd, Kd, Vd))
        o = torch.empty(B, H, d, device="cuda")
        lse = torch.empty(B, H, device="cuda")
        if fused:
            cache.decode_step_fused(q, k, v, o, lse)
        else:
            cache.append_kv(k, v)
            cache.decode_step(q, o, lse)
        torch.cuda.synchronize()
        assert_close(f64(o)[0], ref[m + t], 0, f"step {t}")
        assert abs(lse.item() - ref_lse[m + t, 0]) <= F32_TOL
        # bit-exact ring and sizes against the integer model
        state = oracle.append_kv(state, f64(K[m + t]), f64(V[m + t]), n)
        assert cache.get_t(0) == t + 1 == state["t"]
        assert cache.cache_len(0) == oracle.cache_len(m, n, t + 1)
        assert cache.cache_bytes(0) == oracle.cache_len(m, n, t + 1) * H * d * 2 * 4
        filled = sorted(oracle.ring_outputs(t + 1, n))
        np.testing.assert_array_equal(f64(Ks[0, :, m:])[..., :][:, filled].transpose(1, 0, 2),
                                      state["Kr"][filled])
        np.testing.assert_array_equal(f64(Vs[0, :, m:])[:, filled].transpose(1, 0, 2),
                                      state["Vr"][filled])
    np.testing.assert_array_equal(f64(Ks[0, :, :m]).transpose(1, 0, 2), f64(K[:m]))
    assert cache.sync_status() == 0


def test_tiny_f32_one_shot_prefill(cuda_lib):
    rswa = cuda_lib
    w = workloads.WORKLOADS["tiny_f32"]
    B, H, d, m, n, T = w.batch, w.heads, w.head_dim, w.m, w.n, w.T
    Q, K, V = make_seq([m], T, H, d, 0, seed=0)
    ref, _ = oracle.prefill_attention(f64(Q), f64(K), f64(V), m, n)
    cache = rswa.RswaCache(m, n, H, d, B, rswa.RSWA_F32)
    O = torch.empty_like(Q, device="cuda")
    cache.prefill(Q.cuda(), K.cuda(), V.cuda(), O, [m], T)
    torch.cuda.synchronize()
    assert_close(f64(O), ref, 0, "prefill")
    assert cache.get_t(0) == T
    assert cache.cache_len(0) == oracle.cache_len(m, n, T)
    # ring after a one-shot prefill equals the oracle's
    st = oracle.prefill_cache(f64(K), f64(V), m, n, T)
    Ks, Vs = cache.slabs()
    np.testing.assert_array_equal(f64(Ks[0, :, m:]).transpose(1, 0, 2), st["Kr"])
    np.testing.assert_array_equal(f64(Vs[0, :, m:]).transpose(1, 0, 2), st["Vr"])


# ---------------------------------------------------------------------------
# bf16 prefill over a grid of shapes: tile boundaries, ragged tails, wraps
# ---------------------------------------------------------------------------

PREFILL_CASES = [
    # (m_list, n, T, H, d)
    ([16], 8, 64, 1, 128),
    ([0], 8, 200, 2, 128),
    ([5], 1, 40, 2, 128),
    ([130], 128, 127, 2, 128),
    ([288], 128, 129, 2, 128),
    ([128], 128, 259, 1, 128),
    ([300], 64, 0, 2, 128),
    ([257], 32, 300, 1, 64),
    ([40, 0, 133], 16, 37, 2, 128),
    ([200, 7], 128, 300, 1, 128),
    ([10], 4000, 300, 1, 128),   # n >= T: plain causal attention
    # head_dim 64 on the tensor cores: short units (persistent launch), long
    # units (one per CTA), ragged sequences, grouped heads via test_gqa_prefill
    ([0], 128, 1000, 2, 64),
    ([3000], 128, 500, 2, 64),
    ([40, 0, 133, 700], 16, 37, 3, 64),
    ([1], 1, 1, 1, 64),
]


@pytest.mark.parametrize("case", PREFILL_CASES, ids=lambda c: f"m{c[0]}n{c[1]}T{c[2]}H{c[3]}d{c[4]}")
def test_bf16_prefill(cuda_lib, case):
    rswa = cuda_lib
    m_list, n, T, H, d = case
    Q, K, V = make_seq(m_list, T, H, d, 1, seed=11)
    B = len(m_list)
    cache = rswa.RswaCache(max(m_list), n, H, d, B, rswa.RSWA_BF16)
    O = torch.zeros_like(Q, device="cuda")
    cache.prefill(Q.cuda(), K.cuda(), V.cuda(), O, m_list, T)
    torch.cuda.synchronize()
    assert cache.sync_status() == 0
    refs = oracle_prefill(Q, K, V, m_list, T, n)
    off = 0
    for b, m in enumerate(m_list):
        L = m + T
        assert_close(f64(O[off:off + L]), refs[b][0], 1, f"seq {b}")
        assert cache.get_t(b) == T
        assert cache.cache_len(b) == oracle.cache_len(m, n, T)
        off += L


# ---------------------------------------------------------------------------
# bf16 decode: fused and unfused against prefill rows, ring sentinels
# ---------------------------------------------------------------------------

DECODE_CASES = [
    # (m_list, n, T, H, d)
    ([288], 128, 300, 2, 128),
    ([0], 8, 30, 2, 128),
    ([64, 300, 5], 16, 40, 2, 128),
    ([100], 7, 23, 1, 64),
    ([1500], 128, 140, 1, 128),
    ([300], 2048, 200, 2, 128),   # n >= T: the full-cache (MHA) baseline
    ([64], 512, 300, 2, 128),     # n >= T on the cluster path
    # more than 152 heads in flight: the split-K kernel with its global combine
    # (m_b = 0 sequences have a single chunk and skip the combine)
    ([0 if i % 4 == 0 else 37 * (i % 7) + 3 for i in range(20)], 16, 12, 8, 128),
]


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("case", DECODE_CASES, ids=lambda c: f"m{c[0]}n{c[1]}T{c[2]}")
def test_bf16_decode(cuda_lib, case, fused):
    rswa = cuda_lib
    m_list, n, T, H, d = case
    B = len(m_list)
    Q, K, V = make_seq(m_list, T, H, d, 1, seed=5)
    refs = oracle_prefill(Q, K, V, m_list, T, n)
    offs = np.cumsum([0] + [m + T for m in m_list])
    cache = rswa.RswaCache(max(m_list), n, H, d, B, rswa.RSWA_BF16)
    # prefill the prefixes only (T = 0): pack the prefix rows
    pk = torch.cat([K[offs[b]:offs[b] + m_list[b]] for b in range(B)]).cuda()
    pv = torch.cat([V[offs[b]:offs[b] + m_list[b]] for b in range(B)]).cuda()
    cache.prefill(None, pk, pv, None, m_list, 0)
    got = np.zeros((T, B, H, d))
    lse_got = np.zeros((T, B, H))
    for t in range(T):
        rows = [offs[b] + m_list[b] + t for b in range(B)]
        q, k, v = (x[rows].contiguous().cuda() for x in (Q, K, V))
        o = torch.empty(B, H, d, dtype=torch.bfloat16, device="cuda")
        lse = torch.empty(B, H, device="cuda")
        if fused:
            cache.decode_step_fused(q, k, v, o, lse)
        else:
            cache.append_kv(k, v)
            cache.decode_step(q, o, lse)
        got[t] = f64(o)
        lse_got[t] = f64(lse)
    torch.cuda.synchronize()
    assert cache.sync_status() == 0
    for b, m in enumerate(m_list):
        assert_close(got[:, b], refs[b][0][m:], 1, f"seq {b}")
        assert np.abs(lse_got[:, b] - refs[b][1][m:]).max() <= 1e-3
        assert cache.get_t(b) == T
        assert cache.cache_len(b) == oracle.cache_len(m, n, T)


@pytest.mark.parametrize("fused", [False, True])
def test_reprefill_then_decode_sees_new_prefix(cuda_lib, fused):
    """Decode launches after the first one may load the prefix before their
    dependency wait; the first decode after a new prefill may not.  Prefill
    prefix A, decode three steps, prefill a different prefix B into the same
    cache and decode at once, all enqueued back to back on one stream: every
    step after the second prefill must match the oracle on prefix B."""
    rswa = cuda_lib
    m, n, H, d, T = 288, 128, 10, 128, 4
    cache = rswa.RswaCache(m, n, H, d, 1, rswa.RSWA_BF16)
    seqs = [make_seq([m], T, H, d, 1, seed=s) for s in (21, 22)]
    outs = []
    for Q, K, V in seqs:
        Qc, Kc, Vc = Q.cuda(), K.cuda(), V.cuda()
        cache.prefill(None, Kc[:m], Vc[:m], None, [m], 0)
        o = torch.empty(T, 1, H, d, dtype=torch.bfloat16, device="cuda")
        for t in range(T):
            q, k, v = (x[m + t][None].contiguous() for x in (Qc, Kc, Vc))
            if fused:
                cache.decode_step_fused(q, k, v, o[t])
            else:
                cache.append_kv(k, v)
                cache.decode_step(q, o[t])
        outs.append(o)
    torch.cuda.synchronize()
    assert cache.sync_status() == 0
    for (Q, K, V), o in zip(seqs, outs):
        ref = oracle_prefill(Q, K, V, [m], T, n)[0][0][m:]
        assert_close(f64(o[:, 0]), ref, 1, "after prefill")
    assert cache.get_t(0) == T


BLOCK_CASES = [
    # (m_list, n, T, block sizes in order, H, d)
    ([288], 128, 0, [5, 1, 34, 128, 7, 100], 2, 128),
    ([40, 0, 300], 16, 0, [16, 3, 9, 16], 2, 128),
    ([17], 8, 0, [8, 8, 3], 1, 64),
]


@pytest.mark.parametrize("case", BLOCK_CASES, ids=lambda c: f"m{c[0]}n{c[1]}")
def test_bf16_decode_block(cuda_lib, case):
    """Blocks of consecutive outputs (speculative-verify shape) must equal
    the prefill rows m + t .. m + t + k - 1 of the same sequence."""
    rswa = cuda_lib
    m_list, n, _, blocks, H, d = case
    B = len(m_list)
    T = sum(blocks)
    Q, K, V = make_seq(m_list, T, H, d, 1, seed=9)
    refs = oracle_prefill(Q, K, V, m_list, T, n)
    offs = np.cumsum([0] + [m + T for m in m_list])
    cache = rswa.RswaCache(max(m_list), n, H, d, B, rswa.RSWA_BF16)
    pk = torch.cat([K[offs[b]:offs[b] + m_list[b]] for b in range(B)]).cuda()
    pv = torch.cat([V[offs[b]:offs[b] + m_list[b]] for b in range(B)]).cuda()
    cache.prefill(None, pk, pv, None, m_list, 0)
    t = 0
    for kb in blocks:
        rows = [[offs[b] + m_list[b] + t + i for i in range(kb)] for b in range(B)]
        q, k, v = (torch.stack([x[r] for r in rows]).contiguous().cuda()
                   for x in (Q, K, V))
        o = torch.empty_like(q)
        lse = torch.empty(B, kb, H, device="cuda")
        cache.decode_block(q, k, v, o, lse)
        torch.cuda.synchronize()
        for b, m in enumerate(m_list):
            assert_close(f64(o[b]), refs[b][0][m + t:m + t + kb], 1,
                         f"block at t={t} seq {b}")
            assert np.abs(f64(lse[b]) - refs[b][1][m + t:m + t + kb]).max() <= 1e-3
        t += kb
        for b in range(B):
            assert cache.get_t(b) == t
    assert cache.sync_status() == 0
    with pytest.raises(rswa.RswaError):
        empty = torch.zeros(B, 0, H, d, dtype=torch.bfloat16, device="cuda")
        cache.decode_block(empty, empty, empty, empty)     # block 0


def test_ring_sentinels_bit_exact(cuda_lib):
    """K/V filled with their token position: the ring must hold exactly the
    outputs the integer model names, in the slots it names."""
    rswa = cuda_lib
    m, n, H, d, B = 9, 16, 2, 128, 1
    T0 = 5
    pos = torch.arange(m + 200, dtype=torch.float32)
    K = pos[:, None, None].expand(m + 200, H, d).contiguous()
    V = (-pos)[:, None, None].expand(m + 200, H, d).contiguous()
    cache = rswa.RswaCache(m, n, H, d, B, rswa.RSWA_F32)
    cache.prefill(None, K[:m + T0].cuda(), V[:m + T0].cuda(), None, [m], T0)
    Ks, Vs = cache.slabs()
    q = torch.zeros(B, H, d, device="cuda")
    o = torch.empty(B, H, d, device="cuda")
    for t in range(T0, T0 + 3 * n + 5):
        cache.decode_step_fused(q, K[m + t][None].cuda(), V[m + t][None].cuda(), o)
        torch.cuda.synchronize()
        held = oracle.ring_outputs(t + 1, n)
        ring = Ks[0, 0, m:, 0].cpu().numpy()
        for slot, j in held.items():
            assert ring[slot] == m + j, (t, slot, j)
            assert Vs[0, 1, m + slot, 5].item() == -(m + j)
        np.testing.assert_array_equal(Ks[0, 0, :m, 0].cpu().numpy(), np.arange(m))
        # q = 0: o is the mean of the visible values, exact for position ids
        vis = list(range(m)) + [m + j for j in held.values()]
        assert abs(o[0, 0, 0].item() + np.mean(vis)) < 1e-3


def test_set_t_resume_and_wrap(cuda_lib):
    """Fill the ring with T = n outputs, restore t_b = 4096 + 37 and keep
    decoding: the write slot follows t_b mod n."""
    rswa = cuda_lib
    m, n, H, d, B = 200, 128, 2, 128, 2
    Q, K, V = make_seq([m, m], n, H, d, 1, seed=21)
    cache = rswa.RswaCache(m, n, H, d, B, rswa.RSWA_BF16)
    cache.prefill(None, K.cuda(), V.cuda(), None, [m, m], n)
    t0 = 4096 + 37
    cache.set_t([t0, t0 + 1])
    assert cache.get_t(0) == t0 and cache.get_t(1) == t0 + 1
    L = m + n
    states = [oracle.prefill_cache(f64(K[b * L:(b + 1) * L]), f64(V[b * L:(b + 1) * L]),
                                   m, n, n) for b in range(B)]
    for b in range(B):
        states[b]["t"] = t0 + b   # same ring contents, restored counter
    gen = workloads.qkv(10 * B, H, d, seed=99, dtype=torch.bfloat16)
    for step in range(10):
        q, k, v = (x[step * B:(step + 1) * B].contiguous() for x in gen)
        o = torch.empty(B, H, d, dtype=torch.bfloat16, device="cuda")
        cache.decode_step_fused(q.cuda(), k.cuda(), v.cuda(), o)
        for b in range(B):
            states[b], ro, _ = oracle.decode_step_fused(states[b], f64(q[b]), f64(k[b]),
                                                        f64(v[b]), n)
            assert_close(f64(o[b]), ro, 1, f"step {step} seq {b}")
    Ks, _ = cache.slabs()
    for b in range(B):
        slot = (t0 + b + 9) % n
        np.testing.assert_array_equal(f64(Ks[b, :, m + slot]), f64(gen[1][9 * B + b]))
        assert cache.get_t(b) == t0 + b + 10


def test_empty_cache_decode(cuda_lib):
    rswa = cuda_lib
    cache = rswa.RswaCache(4, 4, 1, 128, 1, rswa.RSWA_BF16)
    q = torch.ones(1, 1, 128, dtype=torch.bfloat16, device="cuda")
    o = torch.full((1, 1, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, 1, device="cuda")
    cache.decode_step(q, o, lse)
    torch.cuda.synchronize()
    assert (o == 0).all() and lse.item() == float("-inf")


# ---------------------------------------------------------------------------
# host-side error paths with a live handle (no GPU fault involved)
# ---------------------------------------------------------------------------

def test_errors_launch_nothing(cuda_lib):
    rswa = cuda_lib
    m, n, H, d = 32, 8, 1, 128
    cache = rswa.RswaCache(m, n, H, d, 1, rswa.RSWA_BF16)
    K = torch.randn(m + 4, H, d, device="cuda").bfloat16()
    cache.prefill(None, K[:m + 4], K[:m + 4], None, [m], 4)
    with pytest.raises(rswa.RswaError) as e:
        cache.prefill(None, K, K, None, [m + 1], 3)          # m_b > capacity
    assert e.value.status == 2
    with pytest.raises(rswa.RswaError) as e:
        cache.prefill(None, K, K, None, [m], -1)             # T < 0
    assert e.value.status == 1
    with pytest.raises(rswa.RswaError) as e:
        cache.prefill(None, K, K, K, [m], 4)                 # O without Q
    assert e.value.status == 1
    rswa.rswa_debug_fail_next_cuda(1)
    with pytest.raises(rswa.RswaError) as e:
        cache.append_kv(K[:1], K[:1])
    assert e.value.status == 5
    assert cache.get_t(0) == 4                               # nothing ran
    h = cache.handle
    cache.close()
    with pytest.raises(rswa.RswaError) as e:
        rswa.rswa_decode_step(h, K[:1], K[:1])
    assert e.value.status == 4


# ---------------------------------------------------------------------------
# grouped heads (H_kv < H) and varlen packed prefill
# ---------------------------------------------------------------------------

def _qkv_gqa(rows, H, Hkv, d, seed, dtype=torch.bfloat16):
    Q = workloads.normal((rows, H, d), 3 * seed, 1.0, dtype)
    K = workloads.normal((rows, Hkv, d), 3 * seed + 1, 1.0, dtype)
    V = workloads.normal((rows, Hkv, d), 3 * seed + 2, 1.0, dtype)
    return Q, K, V


@pytest.mark.parametrize("d", [128, 64])
def test_gqa_prefill(cuda_lib, d):
    rswa = cuda_lib
    H, Hkv, n, T = 8, 2, 64, 150
    m_list = [100, 260]
    rows = sum(m + T for m in m_list)
    Q, K, V = _qkv_gqa(rows, H, Hkv, d, seed=31)
    cache = rswa.RswaCache(max(m_list), n, H, d, len(m_list), rswa.RSWA_BF16,
                           kv_heads=Hkv)
    O = torch.zeros_like(Q, device="cuda")
    cache.prefill(Q.cuda(), K.cuda(), V.cuda(), O, m_list, T)
    torch.cuda.synchronize()
    off = 0
    for b, m in enumerate(m_list):
        L = m + T
        ref, _ = oracle.prefill_attention(f64(Q[off:off + L]), f64(K[off:off + L]),
                                          f64(V[off:off + L]), m, n)
        assert_close(f64(O[off:off + L]), ref, 1, f"seq {b}")
        assert cache.cache_bytes(b) == oracle.cache_len(m, n, T) * Hkv * d * 2 * 2
        off += L


@pytest.mark.parametrize("B,H,Hkv,m0", [
    (1, 8, 2, 40),      # cluster path
    (2, 6, 3, 40),      # cluster path
    (20, 8, 2, 40),     # grouped split-K, 4 query heads per CTA
    (20, 6, 3, 40),     # grouped split-K, 2 query heads per CTA
    (26, 6, 1, 40),     # one KV head (multi-query), 2 per CTA
    (1, 8, 2, 1500),    # few heads, long cache: grouped split-K
    (1, 8, 2, 6000),    # 256-row chunks: each warp's stage ring wraps
])
@pytest.mark.parametrize("fused", [False, True])
def test_gqa_decode(cuda_lib, B, H, Hkv, m0, fused):
    rswa = cuda_lib
    d, n, T = 128, 16, 24
    m_list = [m0 + 23 * b for b in range(B)]
    rows = sum(m + T for m in m_list)
    Q, K, V = _qkv_gqa(rows, H, Hkv, d, seed=33)
    offs = np.cumsum([0] + [m + T for m in m_list])
    cache = rswa.RswaCache(max(m_list), n, H, d, B, rswa.RSWA_BF16, kv_heads=Hkv)
    pk = torch.cat([K[offs[b]:offs[b] + m_list[b]] for b in range(B)]).cuda()
    pv = torch.cat([V[offs[b]:offs[b] + m_list[b]] for b in range(B)]).cuda()
    cache.prefill(None, pk, pv, None, m_list, 0)
    got = np.zeros((T, B, H, d))
    for t in range(T):
        r = [offs[b] + m_list[b] + t for b in range(B)]
        q, k, v = (x[r].contiguous().cuda() for x in (Q, K, V))
        o = torch.empty(B, H, d, dtype=torch.bfloat16, device="cuda")
        if fused:
            cache.decode_step_fused(q, k, v, o)
        else:
            cache.append_kv(k, v)
            cache.decode_step(q, o)
        got[t] = f64(o)
    torch.cuda.synchronize()
    assert cache.sync_status() == 0
    for b, m in enumerate(m_list):
        sl = slice(offs[b], offs[b] + m + T)
        ref, _ = oracle.prefill_attention(f64(Q[sl]), f64(K[sl]), f64(V[sl]), m, n,
                                          rows=list(range(m, m + T)))
        assert_close(got[:, b], ref, 1, f"seq {b}")
        assert cache.get_t(b) == T


@pytest.mark.parametrize("dtype,d", [(1, 64), (0, 128), (0, 64)],
                         ids=["bf16-d64", "f32-d128", "f32-d64"])
@pytest.mark.parametrize("H,Hkv", [(8, 2), (6, 3)], ids=["G4", "G2"])
def test_gqa_decode_dtypes(cuda_lib, dtype, d, H, Hkv):
    """Grouped split-K decode on the CUDA cores, for the element types and
    head sizes the tensor-core kernel does not take: the reduce-scatter loop
    wherever its shape fits, the plain grouped loop for float32 d 128 with
    two heads per CTA."""
    rswa = cuda_lib
    B, n, T = 20, 16, 12
    m_list = [300 + 37 * b for b in range(B)]
    rows = sum(m + T for m in m_list)
    Q, K, V = _qkv_gqa(rows, H, Hkv, d, seed=44, dtype=tdt(dtype))
    offs = np.cumsum([0] + [m + T for m in m_list])
    cache = rswa.RswaCache(max(m_list), n, H, d, B, dtype, kv_heads=Hkv)
    pk = torch.cat([K[offs[b]:offs[b] + m_list[b]] for b in range(B)]).cuda()
    pv = torch.cat([V[offs[b]:offs[b] + m_list[b]] for b in range(B)]).cuda()
    cache.prefill(None, pk, pv, None, m_list, 0)
    got = np.zeros((T, B, H, d))
    lse_got = np.zeros((T, B, H))
    for t in range(T):
        r = [offs[b] + m_list[b] + t for b in range(B)]
        q, k, v = (x[r].contiguous().cuda() for x in (Q, K, V))
        o = torch.empty(B, H, d, dtype=tdt(dtype), device="cuda")
        lse = torch.empty(B, H, device="cuda")
        cache.decode_step_fused(q, k, v, o, lse)
        got[t] = f64(o)
        lse_got[t] = f64(lse)
    torch.cuda.synchronize()
    assert cache.sync_status() == 0
    for b, m in enumerate(m_list):
        sl = slice(offs[b], offs[b] + m + T)
        ref, rl = oracle.prefill_attention(f64(Q[sl]), f64(K[sl]), f64(V[sl]), m, n,
                                           rows=list(range(m, m + T)))
        assert_close(got[:, b], ref, dtype, f"seq {b}")
        assert np.abs(lse_got[:, b] - rl).max() <= (1e-4 if dtype == 0 else 1e-3)
        assert cache.get_t(b) == T


def test_gqa_decode_tc_multitile(cuda_lib):
    """Grouped decode with several 128-key tiles per split-K chunk (48
    sequences x 8 KV heads of ~800 keys give 512-key chunks), so the K/V ring
    wraps, S^T alternates buffers and PV(j-1) overlaps the softmax of tile j.
    Keys planted late in a chunk (q-aligned, large) raise a head's running
    maximum by far more than 2^8 after the first tile, which forces the O^T
    rescale; the outputs must still match the oracle."""
    rswa = cuda_lib
    B, H, Hkv, d, n, T = 48, 32, 8, 128, 128, 3
    per = H // Hkv
    m_list = [700 + 11 * b for b in range(B)]
    rows = sum(m + T for m in m_list)
    Q, K, V = _qkv_gqa(rows, H, Hkv, d, seed=55)
    offs = np.cumsum([0] + [m + T for m in m_list])
    for b in range(0, B, 5):                # spikes in tiles 2 and 3 of chunk 0
        for r, kvh in ((300 + b, b % Hkv), (450 + 2 * b, (b + 3) % Hkv)):
            qv = Q[offs[b] + m_list[b], kvh * per].float()
            K[offs[b] + r, kvh] = (qv / qv.norm() * 40.0).to(torch.bfloat16)
    cache = rswa.RswaCache(max(m_list), n, H, d, B, rswa.RSWA_BF16, kv_heads=Hkv)
    pk = torch.cat([K[offs[b]:offs[b] + m_list[b]] for b in range(B)]).cuda()
    pv = torch.cat([V[offs[b]:offs[b] + m_list[b]] for b in range(B)]).cuda()
    cache.prefill(None, pk, pv, None, m_list, 0)
    got = np.zeros((T, B, H, d))
    lse_got = np.zeros((T, B, H))
    for t in range(T):
        r = [offs[b] + m_list[b] + t for b in range(B)]
        q, k, v = (x[r].contiguous().cuda() for x in (Q, K, V))
        o = torch.empty(B, H, d, dtype=torch.bfloat16, device="cuda")
        lse = torch.empty(B, H, device="cuda")
        cache.decode_step_fused(q, k, v, o, lse)
        got[t] = f64(o)
        lse_got[t] = f64(lse)
    torch.cuda.synchronize()
    assert cache.sync_status() == 0
    for b in [0, 1, 5, 10, 23, 47]:
        m = m_list[b]
        sl = slice(offs[b], offs[b] + m + T)
        ref, rl = oracle.prefill_attention(f64(Q[sl]), f64(K[sl]), f64(V[sl]), m, n,
                                           rows=list(range(m, m + T)))
        assert_close(got[:, b], ref, 1, f"seq {b}")
        assert np.abs(lse_got[:, b] - rl).max() <= 1e-3
        assert cache.get_t(b) == T


def test_gqa_decode_tc_wrapped_two_tile_ring(cuda_lib):
    """A two-tile ring (n = 256) that has wrapped (T = 300 outputs prefilled,
    so slot j mod n holds output j for j = 44 .. 299) behind multi-tile
    512-key prefix chunks; each fused step's new key and value land in a
    slot of the ring chunk's second or first tile.  Three fused steps must
    match the oracle rows m + 300 .. m + 302."""
    rswa = cuda_lib
    B, H, Hkv, d, n, T0, steps = 24, 32, 8, 128, 256, 300, 3
    m_list = [600 + 13 * b for b in range(B)]       # last chunk 1..3 tiles
    L = [m + T0 + steps for m in m_list]
    Q, K, V = _qkv_gqa(sum(L), H, Hkv, d, seed=61)
    offs = np.cumsum([0] + L)
    cache = rswa.RswaCache(max(m_list), n, H, d, B, rswa.RSWA_BF16, kv_heads=Hkv)
    pk = torch.cat([K[offs[b]:offs[b] + m_list[b] + T0] for b in range(B)]).cuda()
    pv = torch.cat([V[offs[b]:offs[b] + m_list[b] + T0] for b in range(B)]).cuda()
    cache.prefill_varlen(None, pk, pv, None, m_list, [T0] * B)
    got = np.zeros((steps, B, H, d))
    for t in range(steps):
        r = [offs[b] + m_list[b] + T0 + t for b in range(B)]
        q, k, v = (x[r].contiguous().cuda() for x in (Q, K, V))
        o = torch.empty(B, H, d, dtype=torch.bfloat16, device="cuda")
        cache.decode_step_fused(q, k, v, o)
        got[t] = f64(o)
    torch.cuda.synchronize()
    assert cache.sync_status() == 0
    for b in [0, 5, 9, 10, 14, 23]:
        m = m_list[b]
        sl = slice(offs[b], offs[b] + L[b])
        ref, _ = oracle.prefill_attention(f64(Q[sl]), f64(K[sl]), f64(V[sl]), m, n,
                                          rows=list(range(m + T0, m + T0 + steps)))
        assert_close(got[:, b], ref, 1, f"seq {b} (m {m})")
        assert cache.get_t(b) == T0 + steps


@pytest.mark.parametrize("dtype", [1, 0], ids=["bf16-tc", "f32"])
def test_gqa_decode_empty_ring(cuda_lib, dtype):
    """decode_step right after a prefix-only prefill (t_b = 0, nothing
    appended): every ring chunk is empty, so the grouped kernels publish
    empty partials for it and the output is attention over the prefix."""
    rswa = cuda_lib
    B, H, Hkv, d, n = 24, 8, 2, 128, 16
    m_list = [200 + 31 * b for b in range(B)]
    rows = sum(m_list)
    Q, K, V = _qkv_gqa(rows + B, H, Hkv, d, seed=66, dtype=tdt(dtype))
    offs = np.cumsum([0] + m_list)
    cache = rswa.RswaCache(max(m_list), n, H, d, B, dtype, kv_heads=Hkv)
    cache.prefill(None, K[:rows].cuda(), V[:rows].cuda(), None, m_list, 0)
    q = Q[rows:rows + B].contiguous().cuda()
    o = torch.empty(B, H, d, dtype=tdt(dtype), device="cuda")
    lse = torch.empty(B, H, device="cuda")
    cache.decode_step(q, o, lse)
    torch.cuda.synchronize()
    assert cache.sync_status() == 0
    for b in [0, 7, 23]:
        st = oracle.prefill_cache(f64(K[offs[b]:offs[b + 1]]), f64(V[offs[b]:offs[b + 1]]),
                                  m_list[b], n, 0)
        ro, rl = oracle.decode_step(st, f64(q[b]), n)
        assert_close(f64(o[b]), ro, dtype, f"seq {b}")
        assert np.abs(f64(lse[b]) - rl).max() <= (1e-4 if dtype == 0 else 1e-3)
        assert cache.get_t(b) == 0


def test_gqa_decode_block(cuda_lib):
    rswa = cuda_lib
    B, H, Hkv, d, n = 2, 8, 4, 128, 32
    m_list = [70, 130]
    blocks = [7, 32, 1, 20]
    T = sum(blocks)
    rows = sum(m + T for m in m_list)
    Q, K, V = _qkv_gqa(rows, H, Hkv, d, seed=35)
    offs = np.cumsum([0] + [m + T for m in m_list])
    cache = rswa.RswaCache(max(m_list), n, H, d, B, rswa.RSWA_BF16, kv_heads=Hkv)
    pk = torch.cat([K[offs[b]:offs[b] + m_list[b]] for b in range(B)]).cuda()
    pv = torch.cat([V[offs[b]:offs[b] + m_list[b]] for b in range(B)]).cuda()
    cache.prefill(None, pk, pv, None, m_list, 0)
    refs = []
    for b, m in enumerate(m_list):
        sl = slice(offs[b], offs[b] + m + T)
        refs.append(oracle.prefill_attention(f64(Q[sl]), f64(K[sl]), f64(V[sl]),
                                             m, n)[0])
    t = 0
    for kb in blocks:
        r = [[offs[b] + m_list[b] + t + i for i in range(kb)] for b in range(B)]
        q, k, v = (torch.stack([x[rr] for rr in r]).contiguous().cuda()
                   for x in (Q, K, V))
        o = torch.empty_like(q)
        cache.decode_block(q, k, v, o)
        torch.cuda.synchronize()
        for b, m in enumerate(m_list):
            assert_close(f64(o[b]), refs[b][m + t:m + t + kb], 1, f"t={t} seq {b}")
        t += kb


def test_varlen_prefill(cuda_lib):
    """Documents of different prefix and output lengths packed in one call,
    each with its own mask; the cache keeps each sequence's own ring."""
    rswa = cuda_lib
    H, d, n = 2, 128, 32
    m_list, t_list = [50, 0, 300, 129], [10, 200, 0, 77]
    rows = sum(m + t for m, t in zip(m_list, t_list))
    Q, K, V = workloads.qkv(rows, H, d, 41, 1.0, torch.bfloat16)
    cache = rswa.RswaCache(max(m_list), n, H, d, len(m_list), rswa.RSWA_BF16)
    O = torch.zeros_like(Q, device="cuda")
    cache.prefill_varlen(Q.cuda(), K.cuda(), V.cuda(), O, m_list, t_list)
    torch.cuda.synchronize()
    Ks, _ = cache.slabs()
    off = 0
    for b, (m, T) in enumerate(zip(m_list, t_list)):
        L = m + T
        ref, _ = oracle.prefill_attention(f64(Q[off:off + L]), f64(K[off:off + L]),
                                          f64(V[off:off + L]), m, n)
        assert_close(f64(O[off:off + L]), ref, 1, f"seq {b}")
        assert cache.get_t(b) == T
        assert cache.cache_len(b) == oracle.cache_len(m, n, T)
        st = oracle.prefill_cache(f64(K[off:off + L]), f64(V[off:off + L]), m, n, T)
        filled = sorted(oracle.ring_outputs(T, n))
        np.testing.assert_array_equal(
            f64(Ks[b, :, max(m_list):])[:, filled].transpose(1, 0, 2),
            st["Kr"][filled])
        off += L
