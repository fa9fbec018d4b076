"""Parity at the benchmark's full sizes, in the launch configuration that
bench.py times, on outputs the oracle computes one by one."""

import numpy as np
import pytest
import torch

import bench
import oracle

pytestmark = pytest.mark.gpu

BF16_MAX, BF16_MEAN = 2e-2, 5e-3


def f64(t):
    return t.detach().double().cpu().numpy()


def check(got, ref, what):
    err = np.abs(np.asarray(got, np.float64) - ref)
    assert np.isfinite(err).all(), what
    assert err.max() <= BF16_MAX, f"{what}: max {err.max():.3e}"
    assert err.mean() <= BF16_MEAN, f"{what}: mean {err.mean():.3e}"


def test_single_page_graph_replay(cuda_lib):
    dev = torch.device("cuda", 0)
    sp = bench.setup_single_page(dev)
    w = sp["w"]
    m, n, T = w.m, w.n, w.T
    s = sp["stream"]
    with torch.cuda.stream(s):
        sp["g_prefill"].replay()
        sp["g_decode"].replay()
    torch.cuda.synchronize()
    # replay once more: every step restarts from an empty ring
    with torch.cuda.stream(s):
        sp["g_prefill"].replay()
        sp["g_decode"].replay()
    torch.cuda.synchronize()
    assert sp["cache"].sync_status() == 0
    Q, K, V = f64(sp["Q"]), f64(sp["K"]), f64(sp["V"])
    ts = [0, 1, 2, 126, 127, 128, 129, 255, 1000, 4097, T - 1]
    ref, _ = oracle.prefill_attention(Q, K, V, m, n, rows=[m + t for t in ts])
    check(f64(sp["Od"][ts, 0]), ref, "decode rows")
    pr = [0, 1, 100, 127, 128, m - 1]
    refp, _ = oracle.prefill_attention(Q, K, V, m, n, rows=pr)
    check(f64(sp["Op"][pr]), refp, "prefix rows")
    assert sp["cache"].get_t(0) == T
    assert sp["cache"].cache_bytes(0) == oracle.cache_len(m, n, T) * 10 * 128 * 2 * 2


def _seq_state(K, V, off, m, n, T):
    return oracle.prefill_cache(f64(K[off:off + m + T]), f64(V[off:off + m + T]),
                                m, n, T)


def test_batched_decode_full(cuda_lib):
    dev = torch.device("cuda", 0)
    bt = bench.setup_batched(dev)
    w = bt["w"]
    B, H, d, n, T = w.batch, w.heads, w.head_dim, w.n, w.T
    q, k, v = (x[:B] for x in bt["steps"])
    o = torch.empty(B, H, d, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B, H, device=dev)
    bt["cache"].decode_step_fused(q, k, v, o, lse)
    torch.cuda.synchronize()
    assert bt["cache"].sync_status() == 0
    offs = np.cumsum([0] + [m + T for m in bt["m_list"]])
    for b in [0, 1, 17, 33, 63]:
        m = bt["m_list"][b]
        st = _seq_state(bt["K"], bt["V"], offs[b], m, n, T)
        st, ro, rl = oracle.decode_step_fused(st, f64(q[b]), f64(k[b]), f64(v[b]), n)
        check(f64(o[b]), ro, f"seq {b} (m={m})")
        assert np.abs(f64(lse[b]) - rl).max() <= 1e-3
        assert bt["cache"].get_t(b) == T + 1
        assert bt["cache"].cache_len(b) == oracle.cache_len(m, n, T + 1)


def test_batched_gqa_decode_full(cuda_lib):
    """The batched GQA extra (B 64, H 32 over 8 KV heads, m ~ U{256..2048},
    ring full) in bench.py's launch configuration, sampled sequences."""
    dev = torch.device("cuda", 0)
    gq = bench.setup_batched_gqa(dev)
    w = gq["w"]
    B, d, n, T, H = w.batch, w.head_dim, w.n, w.T, gq["H"]
    q, k, v = (x[:B] for x in gq["steps"])
    o = torch.empty(B, H, d, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B, H, device=dev)
    gq["cache"].decode_step_fused(q, k, v, o, lse)
    torch.cuda.synchronize()
    assert gq["cache"].sync_status() == 0
    offs = np.cumsum([0] + [m + T for m in gq["m_list"]])
    for b in [0, 7, 31, 63]:
        m = gq["m_list"][b]
        st = _seq_state(gq["K"], gq["V"], offs[b], m, n, T)
        st, ro, rl = oracle.decode_step_fused(st, f64(q[b]), f64(k[b]), f64(v[b]), n)
        check(f64(o[b]), ro, f"seq {b} (m={m})")
        assert np.abs(f64(lse[b]) - rl).max() <= 1e-3
        assert gq["cache"].get_t(b) == T + 1


@pytest.mark.parametrize("T", [256, 100000])
def test_sweep_decode_full(cuda_lib, T):
    dev = torch.device("cuda", 0)
    sw = bench.setup_sweep(dev)
    w = sw["w"]
    B, H, d, m, n = w.batch, w.heads, w.head_dim, w.m, w.n
    sw["cache"].set_t([T] * B)
    q, k, v = (x[:B] for x in sw["steps"])
    o = torch.empty(B, H, d, dtype=torch.bfloat16, device=dev)
    sw["cache"].decode_step_fused(q, k, v, o)
    torch.cuda.synchronize()
    for b in [0, 13, 31]:
        st = _seq_state(sw["K"], sw["V"], b * (m + n), m, n, n)
        st["t"] = T
        st, ro, _ = oracle.decode_step_fused(st, f64(q[b]), f64(k[b]), f64(v[b]), n)
        check(f64(o[b]), ro, f"T={T} seq {b}")
    Ks, _ = sw["cache"].slabs()
    np.testing.assert_array_equal(f64(Ks[5, :, m + T % n]), f64(k[5]))


def test_multipage_prefill_full(cuda_lib):
    dev = torch.device("cuda", 0)
    pf = bench.setup_prefill(dev, layers=1)
    w = pf["w"]
    m, n, T = w.m, w.n, w.T
    L = m + T
    (Q, K, V), cache, O = pf["qkv"][0], pf["caches"][0], pf["outs"][0]
    cache.prefill(Q, K, V, O, [m], T)
    torch.cuda.synchronize()
    assert cache.sync_status() == 0
    rng = np.random.default_rng(0)
    rows = sorted(set([0, 1, 127, 128, 129, 4095, m - 1, m, m + 1, m + 96,
                       m + 127, m + 128, m + 129, 16383, 16384, L - 129, L - 1]
                      + rng.integers(0, L, 16).tolist()))
    ref, _ = oracle.prefill_attention(f64(Q), f64(K), f64(V), m, n, rows=rows)
    check(f64(O[rows]), ref, "multipage rows")
    assert cache.get_t(0) == T
    assert cache.cache_len(0) == m + n


def _sample_rows(L, tile_edges, rng, extra=24):
    rows = set(x for x in tile_edges if 0 <= x < L)
    rows.update(rng.integers(0, L, extra).tolist())
    return sorted(rows)


def test_vanilla_swa_prefill_full(cuda_lib):
    """m = 0, n = 128, 32K rows, 10 heads, as bench.py's vanilla SWA prefill:
    1280 units of 3 key tiles run persistently, 8-9 units per CTA, so every
    cross-unit phase (Q reload, O hand-over) is exercised many times."""
    import workloads
    rswa = cuda_lib
    dev = torch.device("cuda", 0)
    H, d, n, L = 10, 128, 128, 32768
    Q, K, V = workloads.qkv(L, H, d, 100, 1.0, torch.bfloat16, device=dev)
    cache = rswa.RswaCache(0, n, H, d, 1, rswa.RSWA_BF16, device=dev)
    O = torch.empty(L, H, d, dtype=torch.bfloat16, device=dev)
    cache.prefill(Q, K, V, O, [0], L)
    torch.cuda.synchronize()
    assert cache.sync_status() == 0
    rng = np.random.default_rng(1)
    edges = [0, 1, 126, 127, 128, 129, 255, 256, 257, 383, 384, 511, 512,
             152 * 256 - 1, 152 * 256, 152 * 256 + 130, L - 257, L - 129, L - 1]
    rows = _sample_rows(L, edges, rng)
    ref, _ = oracle.prefill_attention(f64(Q), f64(K), f64(V), 0, n, rows=rows)
    check(f64(O[rows]), ref, "vanilla SWA rows")
    assert cache.get_t(0) == L
    assert cache.cache_len(0) == n


def test_varlen_prefill_persistent_rounds(cuda_lib):
    """Packed sequences with short prefixes (units of 3-11 key tiles, mixed
    prefix, diagonal and band tiles): 510 units over one CTA per SM, so CTAs
    cross sequences and unit shapes from one round to the next."""
    import workloads
    rswa = cuda_lib
    dev = torch.device("cuda", 0)
    H, d, n = 10, 128, 128
    m_list = [0, 300, 77, 1000, 5]
    t_list = [3000, 2500, 4000, 1200, 700]
    rows_total = sum(m + t for m, t in zip(m_list, t_list))
    Q, K, V = workloads.qkv(rows_total, H, d, 55, 1.0, torch.bfloat16, device=dev)
    cache = rswa.RswaCache(max(m_list), n, H, d, len(m_list), rswa.RSWA_BF16,
                           device=dev)
    O = torch.empty_like(Q)
    cache.prefill_varlen(Q, K, V, O, m_list, t_list)
    torch.cuda.synchronize()
    assert cache.sync_status() == 0
    rng = np.random.default_rng(2)
    off = 0
    for b, (m, T) in enumerate(zip(m_list, t_list)):
        L = m + T
        edges = [0, 1, 127, 128, 255, 256, m - 1, m, m + 1, m + 127, m + 128,
                 m + 255, m + 256, L - 129, L - 128, L - 1]
        rows = _sample_rows(L, edges, rng, extra=12)
        sl = slice(off, off + L)
        ref, _ = oracle.prefill_attention(f64(Q[sl]), f64(K[sl]), f64(V[sl]), m,
                                          n, rows=rows)
        check(f64(O[sl][rows]), ref, f"seq {b} (m {m}, T {T})")
        assert cache.get_t(b) == T
        off += L
